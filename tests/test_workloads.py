"""The input generator's byte counts (CPU only): the per-expert and per-step
algorithmic bytes the bench divides by, checked against sums worked by hand
from the tensor shapes of the runner page's MonoLayerWeights."""

from mxfp8_moe_decode_gb300 import workloads as W


def test_expert_bytes_by_hand():
    # E4M3 with 32 x 32 scales at H 5120, I 2048: w13 4096 x 5120 + 128 x 160
    # codes, w2 5120 x 2048 + 160 x 64 codes
    assert W.FULL.expert_bytes() == 20_971_520 + 20_480 + 10_485_760 + 10_240 == 31_488_000
    assert W.FULL.shared_bytes() == 31_488_000
    # E2M1 pairs with a code per row per 32 columns: w13 4096 x 2560 + 4096 x 160,
    # w2 5120 x 1024 + 5120 x 64; the shared expert stays E4M3
    assert W.E384_FP4.expert_bytes() == 10_485_760 + 655_360 + 5_242_880 + 327_680 == 16_711_680
    assert W.E384_FP4.shared_bytes() == 31_488_000


def test_step_bytes_by_hand():
    # gate bf16 [E, H] + bias f32 [E] + the shared expert + U routed experts
    assert W.algorithmic_bytes(W.FULL, 8) == 256 * 5120 * 2 + 256 * 4 + 9 * 31_488_000
    assert W.algorithmic_bytes(W.FULL, 8) == 286_014_464
    assert W.algorithmic_bytes(W.E384_FP4, 245) == (384 * 5120 * 2 + 384 * 4 + 31_488_000
                                                    + 245 * 16_711_680)


def test_workload_table():
    wl = W.WORKLOADS
    assert wl["full_m48_uniform"].dims == W.FULL and wl["full_m48_uniform"].tokens == 48
    assert wl["full_m1"].tokens == 1 and wl["full_m16"].tokens == 16
    assert wl["full_e384_fp4_m48"].dims.routed == "e2m1"
    assert all(w.dims.max_tokens == 48 for w in wl.values())
    assert len({(w.name) for w in wl.values()}) == len(wl)
