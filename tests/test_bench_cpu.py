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
    # The default workload streams from HBM as it is; the small configs fit in L2 and
    # rotate over input copies whose total is more than twice the L2.
    big, _ = bench.io_bytes(synth.workload("long_causal_d128"), None)
    small, _ = bench.io_bytes(synth.workload("dec_causal_bf16"), None)
    assert big > bench.L2_BYTES
    assert small <= bench.L2_BYTES
    assert bench.ROTATE_BYTES > 2 * bench.L2_BYTES


def test_profiled_traffic_needs_the_current_source_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    sha = bench.kernel_source_sha()
    (tmp_path / "attn_tc_wl.md").write_text(f"kernel_source_sha: {sha}\ndram_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic("wl") == 1234.0
    (tmp_path / "attn_tc_wl.md").write_text("kernel_source_sha: 0000000000000000\ndram_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic("wl") is None
    assert bench.profiled_traffic("missing") is None
    # A summary that names its kernel's own sources is checked against those.
    srcs = ("head_attention_gb300/csrc/attn_short.cu", "head_attention_gb300/csrc/ptx.cuh")
    (tmp_path / "attn_short_wl2.md").write_text(
        f"kernel_sources: {' '.join(srcs)}\nkernel_source_sha: {bench.kernel_source_sha(srcs)}\n"
        "dram_bytes_per_launch: 99\n")
    assert bench.profiled_traffic("wl2") == 99.0
    (tmp_path / "attn_short_wl2.md").write_text(
        f"kernel_sources: {' '.join(srcs)}\nkernel_source_sha: {sha}\ndram_bytes_per_launch: 99\n")
    assert bench.profiled_traffic("wl2") is None


def test_percentiles_interpolate_linearly():
    p10, p50, p90 = bench.percentiles([5.0, 1.0, 3.0, 2.0, 4.0])
    assert (p10, p50, p90) == (1.4, 3.0, 4.6)
    assert bench.percentiles([]) == (None, None, None)


def test_key_padding_counts_only_valid_rows():
    # Cross-attention: algorithmic bytes read only the first key_lens[b] rows of K and V,
    # and the visible-pair FLOPs use the same lengths; resident bytes stay dense.
    import numpy as np
    w = synth.workload("cross_bf16")
    lens = np.array([64, 256] * (w.B // 2), dtype=np.int32)
    inp = {"key_lens": lens}
    dense_in, dense_alg = bench.io_bytes(w, None)
    bytes_in, bytes_alg = bench.io_bytes(w, inp)
    row = w.h * (w.d_k + w.d_v) * 2
    assert bytes_in == dense_in
    assert dense_alg - bytes_alg == (w.B * w.n_k - int(lens.sum())) * row
    assert bench.visible_pair_flops(w, inp) == 4.0 * w.h * w.d_k * w.n_q * float(lens.sum())


def test_causal_visible_pairs_are_the_lower_triangle():
    w = synth.workload("long_causal_d128")
    n = w.n_q
    assert bench.visible_pair_flops(w, None) == 4.0 * w.B * w.h * w.d_k * n * (n + 1) / 2
    # the defined count halves the dense one
    assert w.attn_flops() == 2.0 * w.B * w.h * w.d_k * n * n


def test_roofline_bound_is_the_larger_roofline_time():
    peaks = {"bf16_tflops": 1923.5, "bf16_tflops_sustained": 1675.1, "hbm_gbs": 6808.2}
    for name, bound in (("long_causal_d128", "tensor"), ("long_causal_d64", "tensor"),
                        ("dec_causal_bf16", "hbm"), ("cross_bf16", "hbm")):
        w = synth.workload(name)
        _, alg = bench.io_bytes(w, None)
        r = bench.roofline_of(w, "k", w.attn_flops(), bench.visible_pair_flops(w, None), alg, 1.0,
                              peaks, "measured")
        assert r["bound"] == bound, name
        assert r["frac"] == round(r["achieved"] / r["peak"], 4)
    # fp32 runs on CUDA cores: FLOPs are held against the fp32 FMA peak
    w = synth.workload("enc_self_f32")
    _, alg = bench.io_bytes(w, None)
    r = bench.roofline_of(w, "k", w.attn_flops(), None, alg, 1.0, peaks, "measured")
    assert r["bound"] in ("alu", "hbm")
    assert r["peak"] != peaks["bf16_tflops"]


class _FakeSampler:
    def __init__(self, samples):
        self.samples = samples

    def summary(self, window):
        t0, t1 = window
        inside = [s for s in self.samples if t0 <= s <= t1]
        return {"sm_mhz": 2000.0 if inside else None, "samples": len(inside), "reasons": []}


def test_clock_record_falls_back_to_the_sustained_leg():
    # A 14 ms timed region holds one sample: the line's clocks come from the sustained
    # leg that follows, and say so; with enough samples the timed region's own are used.
    rec = {"ms_per_step": 0.7, "_clock_window": (0.0, 0.014),
           "sustained": {"seconds": 3.0, "ms_per_step": 0.71, "_clock_window": (0.02, 3.0)}}
    bench.finalize_clocks(rec, _FakeSampler([0.01] + [0.1 * i for i in range(1, 30)]), 20)
    assert rec["clocks"]["samples"] == 29
    assert rec["clocks"]["timed_region_samples"] == 1
    assert "sustained leg" in rec["clocks"]["source"]
    assert rec["sustained"]["ms_x_median_mhz"] == round(0.71 * 2000.0, 2)
    rec2 = {"ms_per_step": 10.0, "_clock_window": (0.0, 1.0)}
    bench.finalize_clocks(rec2, _FakeSampler([0.1 * i for i in range(10)]), 100)
    assert rec2["clocks"]["source"] == "timed steps"


def test_both_arms_name_the_same_config():
    w = synth.workload("long_causal_d128")
    assert bench.config_of(w, 1) == bench.config_of(w, 1)
    assert set(bench.config_of(w, 1)) >= {"workload", "B", "h", "n_q", "n_k", "d", "mask"}


def test_cpu_baseline_compares_the_sampled_units_with_the_gpu_output():
    # A stand-in for the GPU output that differs from the oracle by exactly 0.25 in one
    # element of every unit: the accumulated max is 0.25 and the mean is 0.25 / elements.
    import numpy as np
    import oracle
    w = synth.Workload("tiny", "bf16", B=2, h=2, n_q=16, n_k=16, d_k=8, d_v=8, mask_kind=1, seed=3)
    inp = synth.attn_inputs(w)

    def gpu_head(b, i):
        q, k, v = bench._head_arrays(inp, w, b, i)
        ref = oracle.attn(q, k, v, w.scale, w.mask_kind, None)[0, :, 0, :].copy()
        ref[3, 2] += 0.25
        return ref

    errs = {}
    rate, threads, desc = bench.oracle_sample_rate(w, inp, 10.0, gpu_head=gpu_head, errs=errs)
    assert errs["n"] == w.B * w.h * w.n_q * w.d_v
    assert abs(errs["max"] - 0.25) < 1e-12
    assert abs(errs["sum"] - 0.25 * w.B * w.h) < 1e-9
    assert rate > 0 and threads >= 1
