"""moe_layer_forward_noalloc: the layer on the library's static scratch.

Some callers cannot allocate device memory where they run the layer (a plugin
whose host application owns every device allocation through its own pool, or a
serving loop that must not call cudaMalloc because it can synchronise the
device). This entry point needs no workspace: its intermediates live in a
fixed 24 MiB static device array inside the library. Here it is checked
against moe_layer_forward (caller workspace) on the Mixtral decode batch, bit
for bit, and against the fp64 oracle within the bf16 tolerance, on two calls
in a row with different tokens, so that the second call also shows that the
scratch left by the first does not leak into its result.

This file is collected last (test_zz_*) so that a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_config, make_tokens, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import TOL, assert_status_ok, host_weights

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 24 << 20


@pytest.fixture(scope="module")
def decode_layer():
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 0)
    L = make_config(1)
    dev = {k: getattr(L, k).cuda() for k in ("x", "w_gate", "w1", "w3", "w2")}
    c = CONFIGS[1]
    x2, _ = make_tokens(c["T"], c["d"], c["E"], c["dtype"], seed=77)
    return L, dev, x2.cuda()


def test_noalloc_matches_workspace_entry_on_two_calls(decode_layer):
    L, dev, x2 = decode_layer
    shape = moe.shape_of(dev["x"], dev["w1"])
    assert 0 < moe.moe_workspace_bytes(shape) <= SCRATCH_BYTES
    for x in (dev["x"], x2):
        ref = moe.layer_forward(x, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
        y = torch.full_like(x, float("nan"))
        moe.moe_layer_forward_noalloc(shape, x, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], y)
        torch.cuda.synchronize()
        assert_status_ok()
        # the same kernels in the same order on the same shape: the same bits
        assert torch.equal(y, ref)
        # and, independently of the other entry point, within the bf16 tolerance of the fp64 oracle
        y_ref = oracle.layer_forward(to_f64(x.cpu()), to_f64(L.w_gate), *host_weights(L))["y"]
        got = to_f64(y.cpu())
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - y_ref)) <= TOL["bf16"] * np.max(np.abs(y_ref))


def test_noalloc_rejects_shapes_beyond_its_scratch(decode_layer):
    _, dev, _ = decode_layer
    big = moe.make_shape(64, 4096, 14336, moe.MOE_BF16)
    assert moe.moe_workspace_bytes(big) > SCRATCH_BYTES
    x = torch.zeros((64, 4096), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros_like(x)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_layer_forward_noalloc(big, x, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], y)
    assert e.value.code == moe.MOE_ERR_WORKSPACE
