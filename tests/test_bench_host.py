"""Host-side logic of bench.py that the reported numbers rest on: the roofline's
algorithmic bytes and the backward's bytes per row, derived here by hand from what each
call must move, and the lookup of a recorded DRAM-traffic figure, which holds only for
the sources it was captured on.  No GPU; bench.py is imported, not run."""
import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_bidirectional_bytes_of_the_k128_workload_by_hand():
    # 16 head-rows (B = 2, H = 8) of N = 65536: bf16 Qx, Kx, V read and O written, 128 B each
    # per row; the fp32 mu, rho (K x d) and alpha (K) of the 8 heads read once
    from gaussian_mixture_latent_gb300 import accounting, inputs
    w = inputs.WORKLOADS["bidir_bf16_n65536"]
    assert (w.B, w.H, w.N, w.d, w.K, w.dv) == (2, 8, 65536, 64, 128, 64)
    rows = 16 * 65536
    expected = rows * (4 * 64 * 2) + 8 * 4 * (128 * 64 * 2 + 128)
    assert expected == 537_399_296
    assert accounting.algorithmic_bytes(w.G, w.N, w.d, w.K, w.dv, w.dtype, w.dtype, H=w.H) == expected


def test_headline_step_moves_both_forwards_bytes():
    # the bench step runs the bidirectional and the causal forward over the same inputs:
    # each reads Qx, Kx, V and writes O once (96 head-rows of N = 8192, d = dv = 64, bf16)
    from gaussian_mixture_latent_gb300 import accounting, inputs
    w = inputs.WORKLOADS["causal_bf16_n8192"]
    assert (w.G, w.N, w.d, w.K, w.dv) == (96, 8192, 64, 64, 64)
    one = 96 * 8192 * 4 * 128 + w.H * 4 * (2 * 64 * 64 + 64)
    assert accounting.algorithmic_bytes(w.G, w.N, w.d, w.K, w.dv, w.dtype, w.dtype, H=w.H) == one


def test_backward_bytes_per_row(bench):
    # bf16 Qx, Kx, V, dO read once (4 x 64 x 2 B) and fp32 dQx, dKx, dV written once (3 x 64 x 4 B)
    from gaussian_mixture_latent_gb300 import inputs
    w = inputs.WORKLOADS["causal_bf16_n8192"]
    assert bench.bwd_bytes_per_row(w) == 4 * 64 * 2 + 3 * 64 * 4 == 1280


def test_backward_path_labels_follow_the_library_rule(bench):
    # tensor-core passes: bidirectional bf16 at d = dv = K = 64 with more than one tile per head;
    # the CUDA-core kernels specialised to that shape otherwise; every other shape the general path
    from gaussian_mixture_latent_gb300 import inputs
    w = inputs.WORKLOADS["causal_bf16_n8192"]
    bid = w.replace(causal=False)
    assert bench.bwd_tc_path(bid) and not bench.bwd_simt64_path(bid)
    assert not bench.bwd_tc_path(w) and bench.bwd_simt64_path(w)
    assert not bench.bwd_tc_path(bid.replace(N=128)) and bench.bwd_simt64_path(bid.replace(N=128))
    k128 = inputs.WORKLOADS["bidir_bf16_n65536"]
    assert not bench.bwd_tc_path(k128) and not bench.bwd_simt64_path(k128)


def test_recorded_traffic_holds_only_for_the_sources_it_was_taken_on(bench, monkeypatch):
    path = os.path.join(ROOT, "profiles", "kernel_traffic.txt")
    entries = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert entries, "no recorded traffic"
    kernel, workload, digest, nbytes = entries[0]
    monkeypatch.setattr(bench, "WORKLOAD", workload)
    monkeypatch.setattr(bench, "csrc_hash", lambda k=None: digest)
    assert bench.known_traffic(kernel) == int(nbytes)
    monkeypatch.setattr(bench, "csrc_hash", lambda k=None: "0" * 16)        # sources changed since
    assert bench.known_traffic(kernel) is None
    monkeypatch.setattr(bench, "csrc_hash", lambda k=None: digest)
    monkeypatch.setattr(bench, "WORKLOAD", "another_workload")
    assert bench.known_traffic(kernel) is None


def test_source_hash_follows_the_kernel_sources(bench):
    # a kernel listed with its sources hashes only those files; an unlisted one hashes all of csrc
    assert bench.csrc_hash("tc_causal") != bench.csrc_hash()
    assert bench.csrc_hash("tc_causal") == bench.csrc_hash("tc_causal_seg")
    assert bench.csrc_hash("tc_write") == bench.csrc_hash("tc_read")


def test_whole_job_rate_adds_the_ranks(bench):
    # units per rank x ranks / seconds
    assert bench.whole_job_rate(1000, 4, 2.0) == pytest.approx(1000 * 4 / 2e-3)
