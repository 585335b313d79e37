"""The bench line's roofline arithmetic on CPU: the algorithmic work of each
kernel group at the 1B shape (the byte and FLOP counts the profile summaries
and the design notes quote), the achieved / peak fractions computed from a
time, and the workload names of the configurations."""
import bench
import synth

# the 1B layer as the bench measures it: 311361 TwELL entries, 150 fallback rows
_N, _D, _F, _T, _C, _NNZ, _NFB = 4096, 2048, 8192, 128, 8, 311361, 150


def test_kernel_work_at_the_1b_shape():
    w = bench.kernel_work(_N, _D, _F, _T, _C, _NNZ, _NFB)
    assert w["up_pack"]["bound"] == "tensor" and w["up_pack"]["flops"] == 137438953472.0
    assert w["sddmm"]["flops"] == w["up_pack"]["flops"]
    # the figures quoted beside the ncu captures (dw_walk_1b.md, launches_1b_fwd_bwd.md)
    assert w["dw"]["bytes"] == 170918538
    assert w["spmm"]["bytes"] == 56885248
    assert w["dx"]["bytes"] == 61079552
    assert w["pack"]["bytes"] == w["unpack"]["bytes"] == 76136448
    # the gathers pull one d_model-wide bf16 row per entry (two for the dW walk)
    assert w["spmm"]["l2_gather_bytes"] == _NNZ * _D * 2
    assert w["dw"]["l2_gather_bytes"] == 2 * _NNZ * _D * 2
    assert "l2_gather_bytes" not in w["up_pack"]
    # fallback rows on the tensor cores: 2 d f per row and product
    assert w["fb_down"]["flops"] == 2.0 * _NFB * _D * _F
    assert w["dx_fallback"]["flops"] == 2 * w["fb_down"]["flops"]
    assert w["dw_fallback"]["flops"] == 3 * w["fb_down"]["flops"]


def test_roofline_entry_fractions():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    e = bench.roofline_entry({"bound": "hbm", "bytes": 6e9, "what": "k"}, 2000.0, peaks, "measured")
    assert e["achieved"] == 3000.0 and e["frac"] == 0.5 and e["unit"] == "GB/s"
    e = bench.roofline_entry({"bound": "tensor", "flops": 1e12, "what": "k"}, 1000.0, peaks, "measured")
    assert e["achieved"] == 1000.0 and e["frac"] == 0.5 and e["frac_of_sustained"] == 0.625
    e = bench.roofline_entry({"bound": "hbm", "bytes": 1e9, "l2_gather_bytes": 2e10, "what": "k"}, 1000.0, peaks,
                             "measured")
    assert e["l2_gather_tbs"] == 20.0


def test_workload_names():
    assert bench.workload_name(synth.CONFIGS["1b"]).startswith(
        "1B-scale FFN fwd+bwd: N=4096 d_model=2048 d_ff=8192 T=128 C=8")
    name = bench.workload_name(synth.CONFIGS["train"])
    assert "N=8192" in name and "1% rows at 20%" in name and "lambda 0.0001" in name


def test_cpu_baseline_leg_runs():
    """The bench's CPU leg (the oracle timed on the host cores) on a few rows
    of the small layer: the same call the bench line makes, run here so a
    broken leg fails on CPU."""
    line = bench.cpu_baseline("pr1", rows=16)
    assert line["kind"] == "oracle" and line["unit"] == bench.UNIT and line["value"] > 0
    assert line["cores"] >= 1 and "pr1 layer" in line["sample"]
