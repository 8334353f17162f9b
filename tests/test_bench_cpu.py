"""The benchmark's roofline arithmetic (algorithmic flops and bytes per call), checked
against closed forms for the configurations' shapes, and its JSON contract keys."""
import numpy as np

import bench
from deepseek_v4_sparse_dsa_gb300.synth import Workload


def _shape_only(B, next_n, lens, topk, dtype="bf16", causal=True, gather=False):
    """A Workload carrying only what the roofline arithmetic reads (no tensors)."""
    lens = np.asarray(lens, dtype=np.int32)
    z = np.zeros(0, np.uint8)
    return Workload("shape", B, next_n, lens, causal, topk, dtype, z, None, z, z, None, None, 64,
                    kv_fp4=z if gather else None)


def test_prefill_flops_closed_form():
    # T = K = 16384, causal: query t sees t + 1 keys; 2 * 64 * 128 flops per visible pair
    wl = _shape_only(1, 16384, [16384], 512)
    T = 16384
    assert bench.algorithmic_work(wl)["flops"] == 2 * 64 * 128 * (T * (T + 1) // 2)
    assert abs(bench.algorithmic_work(wl)["flops"] - 2.199e12) / 2.199e12 < 1e-3


def test_fp8_chunked_flops_closed_form():
    # 8192 queries at positions 57344..65535 over 65536 keys
    wl = _shape_only(1, 8192, [65536], 1024, dtype="e4m3", gather=True)
    visible = sum(57344 + i + 1 for i in range(8192))
    assert bench.algorithmic_work(wl)["flops"] == 2 * 64 * 128 * visible
    assert abs(bench.algorithmic_work(wl)["flops"] - 8.246e12) / 8.246e12 < 1e-3
    # gather: 68 B read + 256 B written + 4 B position per selected row
    assert bench.algorithmic_work(wl)["gather_bytes"] == 8192 * 1024 * (68 + 256 + 4)


def test_decode_bytes_read_every_key_once():
    lens = [4096, 65536, 30000]
    wl = _shape_only(3, 1, lens, 512)
    w = bench.algorithmic_work(wl)
    keys = sum(lens) * 128 * 2
    q = 3 * 64 * 128 * 2 + 3 * 64 * 4          # bf16 q rows + fp32 head weights
    out = 3 * 512 * 8 + 3 * 4                  # selections + context lengths
    assert w["fused_bytes"] == keys + q + out
    # two causal queries per sequence read the sequence's keys once
    wl2 = _shape_only(3, 2, lens, 512)
    assert bench.algorithmic_work(wl2)["fused_bytes"] - bench.algorithmic_work(wl)["fused_bytes"] == \
        3 * (64 * 128 * 2 + 64 * 4) + 3 * 512 * 8


def test_e4m3_key_scales_counted():
    wl = _shape_only(1, 1, [1000], 64, dtype="e4m3", causal=False)
    w = bench.algorithmic_work(wl)
    assert w["fused_bytes"] == 1000 * 128 + 1000 * 4 + (64 * 128 + 64 * 4 + 64 * 4) + 64 * 8 + 4


def test_workloads_and_metric_are_named():
    assert set(bench.WORKLOADS) == {"tiny", "flash_decode", "pro_mtp", "prefill", "fp8_chunked"}
    assert bench.HEADLINE == "fp8_chunked"       # the largest configuration that fits one GPU
    assert bench.UNIT == "query-tokens/s"
    peaks = bench.load_peaks()
    assert peaks["hbm_gbs"] > 0 and peaks["bf16_tflops"] > 0 and peaks["source"] in ("measured", "fallback")


def test_roofline_fraction_recomputes_from_the_record():
    # a record's frac is its algorithmic work / its own ms / the peak it names
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0, "source": "measured"}
    wl = _shape_only(1, 8192, [65536], 1024, dtype="e4m3", gather=True)
    w = bench.algorithmic_work(wl)
    r = bench.roofline("tensor", wl, w, 4.0, peaks)
    assert r["peak"] == 3000.0 and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - w["flops"] / 4e-3 / 1e12 / 3000.0) < 1e-12
    wl2 = _shape_only(4, 1, [5000, 6000, 7000, 8000], 512)
    w2 = bench.algorithmic_work(wl2)
    r2 = bench.roofline("hbm", wl2, w2, 0.01, peaks)
    assert r2["unit"] == "GB/s" and abs(r2["frac"] - w2["fused_bytes"] / 1e-5 / 1e9 / 6000.0) < 1e-12


def test_config_is_shared_by_both_arms():
    wl = _shape_only(1, 8192, [65536], 1024, dtype="e4m3", gather=True)
    c = bench.config_of("fp8_chunked", wl, 0, 1)
    assert c["workload"] == "fp8_chunked" and c["topk"] == 1024 and c["dtype"] == "e4m3"
    assert "gather" in c["l2"]                   # the 2 GiB output write flushes L2 every step


def test_attention_work_closed_form():
    # 3 rows x top-4 with 2 padded slots: 10 live rows of 68 B, q bf16 + fp32 out per row,
    # 4 B per slot, the 64 sinks; 4 x 64 x 128 flops per (row, slot) for S and P.V
    from deepseek_v4_sparse_dsa_gb300.synth import AttnBatch
    sel = np.array([[1, 2, -1, 3], [0, 0, 0, 0], [5, -1, 6, 7]], np.int32)
    z = np.zeros(0, np.uint8)
    ab = AttnBatch("shape", 3, 1, np.array([8, 8, 8]), 4, 16, z, sel, z, z, z, z, 0.1)
    nbytes, flops = bench.attn_work(ab)
    assert nbytes == 10 * 68 + 3 * 64 * 128 * (2 + 4) + 12 * 4 + 64 * 4
    assert flops == 4 * 64 * 128 * 3 * 4


def test_next_rows_are_named():
    assert bench.NEXT_NAMES == ("flash_decode_fp4k", "q_rope_quant", "k_hadamard_mxfp4",
                                "sparse_attn_flash_decode", "sparse_attn_pro_mtp", "sparse_attn_fp8_chunked")
