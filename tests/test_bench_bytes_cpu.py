"""The roofline numerator of bench.py (algorithmic bytes per decode step)
against counts made by hand from the model shape (k2-burn README, "Model
shape": hidden 2560, 36 layers, 32 q / 8 KV heads of 128, intermediate 10240,
vocab 250624, untied lm_head, GroupedRMSNorm gains).

Per layer the projections hold 6144 x 2560 (QKV) + 2560 x 4096 (o_proj) +
20480 x 2560 (gate, up) + 2560 x 10240 (down) = 104,857,600 weights in 31,744
rows and 1,638,400 blocks of 64; the lm_head 641,597,440 weights in 250,624
rows and 10,024,960 blocks; 73 norm gains of 2560 bf16 values (2 per layer +
the final one).  One cached position holds K and V of 8 heads x 128 per layer.
"""
import bench
import k2_inputs as ki

S = ki.K2_3P7B
GAINS = 73 * 2560 * 2


def test_bf16_weights_and_kv_bytes():
    by = bench.algorithmic_bytes(S, 4096, "f16", "bf16")
    assert by["weights"] == 36 * 2 * 104_857_600 + 2 * 641_597_440 + GAINS == 8_833_315_840
    assert by["kv"] == 4096 * 36 * 2 * 8 * 128 * 2 == 4096 * 147_456
    assert by["total"] == 9_437_295_616


def test_int8_kv_bytes_include_one_fp16_scale_per_row():
    by = bench.algorithmic_bytes(S, 8192, "i8", "bf16")
    assert by["kv"] == 8192 * 36 * 2 * 8 * (128 + 2) == 8192 * 74_880


def test_fp8_one_byte_per_weight_and_a_scale_per_row():
    by = bench.algorithmic_bytes(S, 4096, "f16", "f8")
    per_layer = 104_857_600 + 4 * 31_744
    lm_head = 641_597_440 + 4 * 250_624
    assert by["weights"] == 36 * per_layer + lm_head + GAINS == 4_422_418_432


def test_int4_half_a_byte_per_weight_and_a_scale_per_64():
    by = bench.algorithmic_bytes(S, 4096, "f16", "q4")
    per_layer = 104_857_600 // 2 + 4 * 1_638_400
    lm_head = 641_597_440 // 2 + 4 * 10_024_960
    assert by["weights"] == 36 * per_layer + lm_head + GAINS == 2_484_638_720
