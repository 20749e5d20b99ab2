"""The roofline byte/FLOP helpers reproduce the cost arithmetic printed on
"Batch invariance and reproducible inference" (Llama-3-8B on an H100)."""
import json
import os

from invariant_fixed_order_gb300 import roofline
from invariant_fixed_order_gb300.config import LLAMA3_8B


def test_cost_arithmetic_matches_page(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "cost_arithmetic.json")))
    cfg = LLAMA3_8B
    kv = roofline.kv_bytes_per_layer(cfg, 2560)
    assert kv == 2 * 2560 * 8 * 128 * 2
    assert round(kv / 1e6, 1) == g["kv_bytes_per_layer_s2560_MB"]
    assert round(kv * 32 / 1e6) == g["kv_bytes_32_layers_s2560_MB"]
    w = roofline.step_weight_bytes(cfg)
    assert round(w / 1e9, 1) == g["step_weights_GB"]
    assert round(w / (g["hbm_TBps_h100"] * 1e12) * 1e3, 2) == g["step_ms_bs1"]
    assert round(kv * 32 / (g["hbm_TBps_h100"] * 1e12) * 1e3, 2) == g["attention_ms_s2560"]
    qkv = roofline.qkv_weight_bytes(cfg)
    assert round(qkv / 1e6, 1) == g["qkv_weights_MB"]
    M = g["qkv_padded_M"]
    fl = roofline.gemm_flops(M, cfg.qkv_dim, cfg.d)
    assert round(fl / 1e9, 2) == g["qkv_padded_GFLOP"]
    assert roofline.gemm_weight_intensity(M, cfg.qkv_dim, cfg.d) == g["qkv_padded_intensity"]
    assert g["qkv_padded_intensity"] < g["h100_ridge_flop_per_byte"]
    assert round(qkv / (g["hbm_TBps_h100"] * 1e12) * 1e6, 1) == g["qkv_memory_us"]
    assert round(fl / (g["h100_bf16_TFLOPs"] * 1e12) * 1e6, 1) == g["qkv_compute_us"]


def test_layer_bytes_8b():
    cfg = LLAMA3_8B
    # 436.2 MB of GEMM weights per layer (qkv 50.3 + o 33.6 + gate/up 234.9 + down 117.4)
    assert round(roofline.layer_weight_bytes(cfg) / 1e6, 1) == 436.2
