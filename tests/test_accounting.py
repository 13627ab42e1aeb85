"""Host-side accounting that the roofline figures rest on (no GPU): the
algorithmic bytes of a step are the needed logit rows, each read once --
(2L+1) rows of V logits for a sampled request (target rows 0..L, draft rows
0..L-1) and (L+1) for a greedy one -- and the workloads' temperature recipe
gives the sampled / greedy split those bytes depend on."""
import torch

import workloads


def _bytes(T, L, V, esize):
    return workloads.algorithmic_bytes(torch.tensor(T, dtype=torch.float32),
                                       torch.tensor(L, dtype=torch.int32), V, esize)


def test_bytes_of_the_fixed_length_workloads():
    # B=32, K=8, V=151936 bf16, all sampled: 32 * 17 rows of 303,872 bytes
    assert _bytes([1.0] * 32, [8] * 32, 151936, 2) == 165_306_368
    # B=128, K=16, V=151936 bf16, T=0.8: 128 * 33 rows
    assert _bytes([0.8] * 128, [16] * 128, 151936, 2) == 1_283_555_328
    # B=512, K=8, V=201088 bf16, 128 greedy (9 rows) and 384 sampled (17 rows)
    T = [0.0] * 128 + [0.5] * 384
    assert _bytes(T, [8] * 512, 201088, 2) == (128 * 9 + 384 * 17) * 402_176 == 3_088_711_680


def test_bytes_of_a_scheduled_batch():
    # sum L = 1283 over 256 sampled requests of V=128256 bf16: (2 * 1283 + 256) rows
    L = [5] * 255 + [1283 - 5 * 255]
    assert _bytes([0.7] * 256, L, 128256, 2) == (2 * 1283 + 256) * 256_512 == 723_876_864


def test_greedy_rules_follow_the_temperature():
    # T <= 0, NaN, inf and subnormal temperatures are greedy (L + 1 rows); fp32 rows are 4 bytes
    T = [0.0, -1.0, float("nan"), float("inf"), 1e-40, 1e-30, 2.0]
    L = [3] * len(T)
    greedy_rows, sampled_rows = 4, 7
    want = (5 * greedy_rows + 2 * sampled_rows) * 1000 * 4
    assert _bytes(T, L, 1000, 4) == want
    # L = 0: the step degenerates to one draw (sampled) or one argmax (greedy): one row each
    assert _bytes([1.0, 0.0], [0, 0], 64, 4) == 2 * 64 * 4


def test_mixed_temperature_recipe():
    """The B=512 workload's split: exactly a quarter greedy (T = 0), the others
    in (0, 1.2]; a shrunk batch keeps the proportion."""
    for B in (512, 64):
        t = workloads.workload_temperatures(4, B, device="cpu")
        assert t.shape == (B,) and t.dtype == torch.float32
        assert int((t == 0).sum()) == B // 4
        pos = t[t != 0]
        assert bool(((pos > 0) & (pos <= 1.2)).all())
    # the fixed-temperature workloads
    assert bool((workloads.workload_temperatures(2, 128, device="cpu") == 0.8).all())
