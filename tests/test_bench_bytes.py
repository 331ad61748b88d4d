"""The algorithmic byte counts behind bench.py's GB/s and roofline figures,
pinned to sums worked out by hand from the workload shapes (not re-typed from
bench.py's formulas).

KIVI INT4 (batch 8 x 8 KV heads, T 8192, d 128, groups of 64, 128 residual
tokens, asymmetric with bf16 scale and zero), K and V together:
 - bf16 source 2 x 134,217,728 B;
 - codes 2 x 33,030,144 B (8064 quantized tokens x 64 B per row);
 - metadata 2 x 4,128,768 B (K: 126 groups x 128 channels, V: 8064 tokens x 2
   groups; 2 B scale + 2 B zero per group, over 64 slices);
 - residual 2 x 2,097,152 B.
 quantize reads the source and writes the rest: 268,435,456 + 78,512,128.
 The statistics read the source, the codes and the metadata (the residual's
 error is zero by construction).
H2O / SnapKV (32 heads, 64 history rows, T 131072, float32 history; budget
2048; K and V rows of 128 bf16): the history rows read (all 64, or the last 32),
the int32 keep set written, and the kept K and V rows read and written.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_kivi_bytes():
    kb = _bench().kivi_bytes()
    src, codes, meta, resid = 2 * 134_217_728, 2 * 33_030_144, 2 * 4_128_768, 2 * 2_097_152
    assert kb["quantize"] == src + codes + meta + resid == 346_947_584
    assert kb["dequantize"] == 346_947_584
    assert kb["error_stats"] == src + codes + meta == 342_753_280


def test_eviction_bytes():
    eb = _bench().evict_bytes()
    hist_all, hist_obs = 32 * 64 * 131_072 * 4, 32 * 32 * 131_072 * 4
    keep = 32 * 2048 * 4
    rows = 2 * (2 * 32 * 2048 * 128 * 2)                    # K and V, read + write
    assert eb["h2o_select"] == hist_all + keep == 1_074_003_968
    assert eb["snapkv_select"] == hist_obs + keep == 537_133_056
    assert eb["h2o_compact"] == eb["snapkv_compact"] == rows == 67_108_864
    assert eb["h2o_select"] + eb["h2o_compact"] == 1_141_112_832
    assert eb["snapkv_select"] + eb["snapkv_compact"] == 604_241_920


def test_fullmodel_and_sweep_row_bytes():
    """Full-model INT8 (32 layers x 8192 tokens x 4096 channels, K and V):
    4,294,967,296 B of bf16 read, 2,147,483,648 B of codes and 262,144 fp32
    scales (1,048,576 B) written -- 6,443,499,520 B per op.  Sweep (16 x 8
    slices x 32768 tokens x 128 channels, K and V = 1,073,741,824 numbers):
    2,147,483,648 B read; INT4 g 64 writes 536,870,912 B of codes and
    33,554,432 B of bf16 scales, INT2 g 64 268,435,456 + 33,554,432 B."""
    bn = _bench()
    fm = bn.fullmodel_bytes()
    assert fm["quantize"] == fm["dequantize"] == fm["error_stats"] == 6_443_499_520
    assert bn.sweep_bytes(4, 64)["quantize"] == 2_147_483_648 + 570_425_344 == 2_717_908_992
    assert bn.sweep_bytes(2, 64)["dequantize"] == 2_147_483_648 + 301_989_888
