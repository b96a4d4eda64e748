"""gma_forward_multi: independent forwards in one request, the causal scan (one CTA per
head) on a second stream beside the other calls.  Every output is checked against the
fp64 oracle (the forward of section 3.3, Eq. 5-8, and of section 3.5, Eq. 6b / 8b) and
against gma_forward on the same inputs: bitwise where the request runs the call's plan
unchanged, and to within the rounding of the key-side partial sums where a
bidirectional call's write kernel ran on the SMs the scan left free."""
import numpy as np
import pytest

from gaussian_mixture_latent_gb300 import inputs
from tests._util import TOL, head_rel_err, oracle_head, to_device, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

THREADS = 16


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def device_inputs(x):
    return {n: to_device(x[n]) for n in ("Qx", "Kx", "V", "mu", "rho", "alpha")}


def call(w, d, causal, **kw):
    c = dict(Qx=d["Qx"], Kx=d["Kx"], V=d["V"], mu=d["mu"], rho=d["rho"], pi_logits=d["alpha"], eps=w.eps,
             causal=causal, var_floor=w.var_floor)
    c.update(kw)
    return c


def single(w, d, causal):
    import gaussian_mixture_latent_gb300 as gma
    out = gma.gma_forward(d["Qx"], d["Kx"], d["V"], d["mu"], d["rho"], d["alpha"], eps=w.eps, causal=causal,
                          var_floor=w.var_floor)
    torch.cuda.synchronize()
    assert gma.gma_get_status() == 0
    return out


def oracle_check(w, x, out, heads):
    from concurrent.futures import ThreadPoolExecutor
    got = to_f64(out).reshape(w.G, w.N, w.dv)
    with ThreadPoolExecutor(THREADS) as ex:
        refs = list(ex.map(lambda g: oracle_head(w, x, g), heads))
    worst = max(head_rel_err(got[g], r) for g, r in zip(heads, refs))
    assert worst <= TOL[w.dtype], (w.name, worst)
    return worst


def close_to(a, b, w):
    """Normwise per-head difference of two bf16 outputs of the same forward whose key-side
    memories were summed over different row splits: the fp32 sums differ in the last
    bits, which can move a bf16 rounding of the memory operand or of an output by one
    unit (2^-8 relative); the bound allows twice that."""
    ga = to_f64(a).reshape(w.G, w.N, w.dv)
    gb = to_f64(b).reshape(w.G, w.N, w.dv)
    worst = max(head_rel_err(ga[g], gb[g]) for g in range(w.G))
    assert worst <= 2 ** -7, (w.name, worst)
    return worst


def test_bidirectional_and_causal_side_by_side_at_full_size():
    # the 96-head N = 8192 workload: the scan holds 96 SMs, the bidirectional write runs on
    # the other 56, its read spreads over every SM once the scan is done
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.WORKLOADS["causal_bf16_n8192"]
    x = inputs.gen_all(w)
    d = device_inputs(x)
    ref_b, ref_c = single(w, d, False), single(w, d, True)
    aux = torch.cuda.Stream()
    ob, oc = gma.gma_forward_multi([call(w, d, False), call(w, d, True)], aux_stream=aux, check_status=True)
    assert torch.equal(oc, ref_c)
    diff = close_to(ob, ref_b, w)
    wb = w.replace(causal=False)
    err_b = oracle_check(wb, x, ob, list(range(w.G)))
    err_c = oracle_check(w, x, oc, [0, 31, 64, 95])
    print(f"bidirectional vs gma_forward {diff:.2e}, vs oracle {err_b:.2e}; causal vs oracle {err_c:.2e}")
    # the same request again gives the same bits
    ob2, oc2 = gma.gma_forward_multi([call(w, d, False), call(w, d, True)], aux_stream=aux, check_status=True)
    assert torch.equal(ob2, ob) and torch.equal(oc2, oc)


def test_without_an_auxiliary_stream_the_calls_run_as_gma_forward_does():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("multi_seq", B=2, H=48, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=5)
    x = inputs.gen_all(w)
    d = device_inputs(x)
    ref_b, ref_c = single(w, d, False), single(w, d, True)
    ob, oc = gma.gma_forward_multi([call(w, d, False), call(w, d, True)], check_status=True)
    assert torch.equal(ob, ref_b) and torch.equal(oc, ref_c)
    # the main stream passed as the auxiliary one: no second lane either
    s = torch.cuda.current_stream()
    ob, oc = gma.gma_forward_multi([call(w, d, False), call(w, d, True)], stream=s, aux_stream=s, check_status=True)
    assert torch.equal(ob, ref_b) and torch.equal(oc, ref_c)


def test_mixed_request_every_path_and_an_empty_call():
    # a per-head causal scan (96 heads, short rows) beside: the bidirectional K = 64 and
    # K = 128 tensor-core paths (write on the free SMs), the fp32 CUDA-core causal path,
    # the segment-parallel causal scan, and an empty call
    import gaussian_mixture_latent_gb300 as gma
    wl = [
        inputs.Workload("m_scan", B=2, H=48, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=6),
        inputs.Workload("m_bidir64", B=2, H=48, N=300, d=64, K=64, dv=64, dtype="bf16", causal=False, seed=7),
        inputs.Workload("m_bidir128", B=1, H=2, N=777, d=64, K=128, dv=64, dtype="bf16", causal=False, seed=8),
        inputs.Workload("m_f32", B=1, H=2, N=333, d=16, K=8, dv=32, dtype="f32", causal=True, seed=9),
        inputs.Workload("m_seg", B=1, H=3, N=5000, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=10),
        inputs.Workload("m_empty", B=1, H=2, N=0, d=64, K=64, dv=64, dtype="bf16", causal=False, seed=11),
    ]
    xs = [inputs.gen_all(w) for w in wl]
    ds = [device_inputs(x) for x in xs]
    refs = [single(w, d, w.causal) if w.N > 0 else None for w, d in zip(wl, ds)]
    aux = torch.cuda.Stream()
    outs = gma.gma_forward_multi([call(w, d, w.causal) for w, d in zip(wl, ds)], aux_stream=aux,
                                 check_status=True)
    for w, x, o, r in zip(wl, xs, outs, refs):
        if w.N == 0:
            assert o.numel() == 0
            continue
        if w.causal:
            assert torch.equal(o, r), w.name          # causal plans run unchanged
        else:
            close_to(o, r, w)
        err = oracle_check(w, x, o, list(range(w.G)))
        print(f"{w.name}: max relative error {err:.2e}")


def test_events_are_recorded_on_the_stream_of_their_call():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("m_ev", B=2, H=48, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=12)
    d = device_inputs(inputs.gen_all(w))
    aux = torch.cuda.Stream()
    ev = {c: [torch.cuda.Event(enable_timing=True) for _ in range(8)] for c in (False, True)}
    for e in ev[False] + ev[True]:
        e.record()
    gma.gma_forward_multi([call(w, d, False, events=ev[False]), call(w, d, True, events=ev[True])],
                          aux_stream=aux, check_status=True)
    torch.cuda.synchronize()
    # the causal call is the single launch of the scan; the bidirectional call has four
    assert ev[True][0].elapsed_time(ev[True][1]) > 0
    assert all(ev[False][2 * i].elapsed_time(ev[False][2 * i + 1]) > 0 for i in range(4))


def test_a_request_captured_in_a_cuda_graph_replays_the_same_results():
    import gaussian_mixture_latent_gb300 as gma
    w = inputs.Workload("m_graph", B=2, H=48, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=13)
    d = device_inputs(inputs.gen_all(w))
    aux = torch.cuda.Stream()
    ob = torch.empty(w.B, w.H, w.N, w.dv, dtype=torch.bfloat16, device="cuda")
    oc = torch.empty_like(ob)
    calls = [call(w, d, False, out=ob), call(w, d, True, out=oc)]
    gma.gma_forward_multi(calls, aux_stream=aux, check_status=True)      # workspace allocated before capture
    eb, ec = ob.clone(), oc.clone()
    ob.zero_(); oc.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gma.gma_forward_multi(calls, stream=s, aux_stream=aux)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ob, eb) and torch.equal(oc, ec)


def test_several_scans_and_several_other_calls_in_one_request():
    # two per-head causal scans (the auxiliary lane runs them in order) beside two
    # bidirectional calls and a cross-shaped pair of problems of different lengths, with
    # events on every call: every output against gma_forward (bitwise for the scans and the
    # unbudgeted calls, within the partial-sum rounding for the budgeted writes) and the oracle
    import gaussian_mixture_latent_gb300 as gma
    wl = [
        inputs.Workload("s_scan_a", B=2, H=48, N=256, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=21),
        inputs.Workload("s_bidir_a", B=1, H=40, N=700, d=64, K=64, dv=64, dtype="bf16", causal=False, seed=22),
        inputs.Workload("s_scan_b", B=1, H=80, N=300, d=64, K=64, dv=64, dtype="bf16", causal=True, seed=23),
        inputs.Workload("s_bidir_b", B=2, H=3, N=1000, d=64, K=128, dv=64, dtype="bf16", causal=False, seed=24),
    ]
    xs = [inputs.gen_all(w) for w in wl]
    ds = [device_inputs(x) for x in xs]
    refs = [single(w, d, w.causal) for w, d in zip(wl, ds)]
    aux = torch.cuda.Stream()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in wl]
    for e in sum(evs, []):
        e.record()
    outs = gma.gma_forward_multi([call(w, d, w.causal, events=e) for w, d, e in zip(wl, ds, evs)], aux_stream=aux,
                                 check_status=True)
    for w, x, o, r in zip(wl, xs, outs, refs):
        if w.causal:
            assert torch.equal(o, r), w.name
        else:
            close_to(o, r, w)
        err = oracle_check(w, x, o, list(range(w.G)))
        print(f"{w.name}: max relative error {err:.2e}")
    torch.cuda.synchronize()
    assert all(e[0].elapsed_time(e[1]) > 0 for e in evs)
