"""The bench's algorithmic byte and work model -- the numerator of every
roofline fraction it reports -- against closed forms of the layer's formats:
a Q8_0 row of K weights is K code bytes plus K/32 fp16 scales, a 2-bit row K/4
code bytes plus the scales, an e2m1 row K/2 plus the scales; each selected
expert and the shared expert are read once per call."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth  # noqa: E402


def test_row_bytes_per_format():
    for K in (128, 2048, 6144):
        assert bench.row_bytes(synth.FMT_Q8_0, K) == K + K // 16
        assert bench.row_bytes(synth.FMT_Q2S, K) == K // 4 + K // 16
        assert bench.row_bytes(synth.FMT_E2M1, K) == K // 2 + K // 16


def test_decode_layer_reads_nine_experts_of_40_mb():
    spec = synth.GLM_LAYER
    per_expert = 3 * spec.f * spec.d * 17 // 16  # gate, up, down at 1.0625 B a weight
    assert per_expert == 40_108_032
    b = bench.stage_bytes(spec, 1, [1] * spec.k)  # 8 routed experts, one row each
    assert b["total"] == 9 * per_expert == 360_972_288
    assert b["decode_fused"] == b["total"]
    assert b["gateup"] == 9 * 2 * spec.f * spec.d * 17 // 16
    assert b["down"] == 9 * spec.d * spec.f * 17 // 16
    assert b["gateup_tc"] == b["down_tc"] == 0


def test_shared_expert_is_counted_once_whatever_the_rows():
    spec = synth.GLM_LAYER
    one = bench.stage_bytes(spec, 1, [1] * 8)["total"]
    many = bench.stage_bytes(spec, 16, [2] * 64)["total"]  # 64 experts, 2 rows each
    per_expert = 3 * spec.f * spec.d * 17 // 16
    assert one == 9 * per_expert
    assert many == 65 * per_expert  # row counts do not change the bytes


def test_two_bit_layer_bytes():
    spec = synth.Q2_LAYER
    routed = 3 * spec.f * spec.d * 5 // 16  # 0.3125 B a weight: 2 bits + fp16/32
    shared = 3 * spec.f_shared * spec.d * 17 // 16
    assert routed == 5_898_240 and shared == 20_054_016
    b = bench.stage_bytes(spec, 64, [3] * 100)
    assert b["total"] == 100 * routed + shared


def test_rows_above_the_threshold_go_to_the_tensor_stages():
    spec = synth.GLM_LAYER
    per_gu = 2 * spec.f * spec.d * 17 // 16
    per_dn = spec.d * spec.f * 17 // 16
    counts = [7, 6, 20, 1]
    b = bench.stage_bytes(spec, 512, counts, tc_rows=6)
    # experts with 7 and 20 rows and the shared expert (512 rows) on the tensor cores
    assert b["gateup_tc"] == 3 * per_gu and b["down_tc"] == 3 * per_dn
    assert b["gateup"] == 2 * per_gu and b["down"] == 2 * per_dn
    # fewer tensor-core gate/up tiles than SMs: every expert on the GEMV
    tiles = bench.tc_tiles(spec, 512, counts, 6)
    assert tiles == (spec.f // 128) * (1 + 1 + 8)  # 7 and 20 rows: one 64-row tile each; shared 512 rows: 8
    b2 = bench.stage_bytes(spec, 512, counts, tc_rows=6, sm_count=tiles + 1)
    assert b2["gateup_tc"] == 0 and b2["gateup"] == 5 * per_gu


def test_macs_count_rows_times_weights():
    spec = synth.GLM_LAYER
    m = bench.stage_macs(spec, 2, [1, 2])
    rows = 1 + 2 + 2  # two routed experts and the shared expert's two tokens
    assert m["gateup"] == 2 * spec.f * spec.d * rows
    assert m["down"] == spec.d * spec.f * rows


def test_unit_fractions_at_the_peak_rates():
    # a stage that issues exactly the dp4a peak (152 SMs x 64 a clock at
    # 2070 MHz) for 1 ms, and a tensor stage at exactly 1000 TFLOP/s
    dp4a_per_ms = 152 * bench.DP4A_PER_SM_CLK * 2070e6 * 1e-3
    macs = {"gateup": 4 * dp4a_per_ms, "down": 2 * dp4a_per_ms,
            "gateup_tc": 1000e12 * 1e-3 / 2, "down_tc": 0}
    stage_ms = {"gateup": 1.0, "down": 1.0, "gateup_tc": 1.0, "down_tc": 1.0}
    f = bench.unit_fractions(macs, stage_ms, 152, 2070.0, 2000.0)
    assert f["gateup_dp4a_frac"] == 1.0 and f["down_dp4a_frac"] == 0.5
    assert f["gateup_tc_tensor_frac"] == 0.5
    assert "down_tc_tensor_frac" not in f  # no work on that stage


def test_both_arms_name_the_workload_alike():
    spec, T, _ = synth.WORKLOADS["decode_t1"]
    desc = bench.workload_desc("decode_t1", spec, T)
    assert desc == ("decode_t1: T=1, E=256, top_k=8, d=6144, f=2048, f_shared=2048, fmt=Q8_0, "
                    "s=2.5, zipf_beta=0.4")
    line = bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1",
                                                 "--warmup", "0"]))
    assert line["config"]["workload"] == desc
    spec4, T4, _ = synth.WORKLOADS["fp4_t64"]
    assert "fmt=E2M1" in bench.workload_desc("fp4_t64", spec4, T4)
