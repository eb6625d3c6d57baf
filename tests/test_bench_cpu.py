"""Host-side logic of bench.py: byte accounting, the L2-flush constants and the
rule that profiled DRAM traffic is reported only for the current kernel source."""

import bench
from synth import inputs as synth


def test_io_bytes_attention_counts_each_tensor_once():
    w = synth.workload("long_causal_d128")
    esize = 2
    q = w.B * w.n_q * w.h * w.d_k * esize
    kv = w.B * w.n_k * w.h * (w.d_k + w.d_v) * esize
    o = w.B * w.n_q * w.h * w.d_v * esize
    bytes_in, bytes_alg = bench.io_bytes(w, None)
    assert bytes_in == q + kv
    assert bytes_alg == q + kv + o


def test_default_workload_exceeds_l2_and_small_ones_do_not():
    # The default workload streams from HBM without a flush; the small configs
    # fit in L2 and are timed with a flush that is itself larger than L2.
    big, _ = bench.io_bytes(synth.workload("long_causal_d128"), None)
    small, _ = bench.io_bytes(synth.workload("dec_causal_bf16"), None)
    assert big > bench.L2_BYTES
    assert small <= bench.L2_BYTES
    assert bench.FLUSH_BYTES > bench.L2_BYTES


def test_profiled_traffic_needs_the_current_source_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    sha = bench.kernel_source_sha()
    (tmp_path / "attn_tc_wl.md").write_text(f"kernel_source_sha: {sha}\ndram_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic("wl") == 1234.0
    (tmp_path / "attn_tc_wl.md").write_text("kernel_source_sha: 0000000000000000\ndram_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic("wl") is None
    assert bench.profiled_traffic("missing") is None
