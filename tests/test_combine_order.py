"""The fused combine rests on one property of IEEE fp32 addition: two operands give the same sum in either
order, signed zeros, subnormals and overflow included. The down projection's finishing slot computes
own + other while the separate pass computes y_slot[r0] + y_slot[r1]; whichever slot is r0, the bits
of y must agree. Checked here on the host with numpy's fp32 arithmetic (round to nearest even), and
for the bf16 rounding that follows."""
import numpy as np
import torch


def _specials():
    f = np.float32
    return np.array([0.0, -0.0, 1.0, -1.0, f(2.0) ** -149, -(f(2.0) ** -149), f(2.0) ** -126,
                     np.finfo(np.float32).max, -np.finfo(np.float32).max, 1e-30, -1e-30, 3.0e38, -3.0e38],
                    dtype=np.float32)


def test_fp32_addition_of_two_operands_is_commutative_bitwise():
    rng = np.random.default_rng(0)
    a = (rng.standard_normal(200_000) * np.exp(rng.uniform(-40, 40, 200_000))).astype(np.float32)
    b = (rng.standard_normal(200_000) * np.exp(rng.uniform(-40, 40, 200_000))).astype(np.float32)
    s = _specials()
    a = np.concatenate([a, np.repeat(s, s.size)])
    b = np.concatenate([b, np.tile(s, s.size)])
    with np.errstate(over="ignore"):
        ab, ba = a + b, b + a
    assert np.array_equal(ab.view(np.uint32), ba.view(np.uint32))


def test_bf16_rounding_of_the_sum_is_the_same_either_way():
    rng = np.random.default_rng(1)
    a = torch.from_numpy(rng.standard_normal(100_000).astype(np.float32))
    b = torch.from_numpy(rng.standard_normal(100_000).astype(np.float32))
    assert torch.equal((a + b).to(torch.bfloat16), (b + a).to(torch.bfloat16))
