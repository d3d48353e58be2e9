"""Several handles and the allocation-free call in one process, launching the
same kernel function with different shared-memory layouts: a smaller shape
created (or stepped without a handle) after a larger one must not stop the
larger handle's next launch. The per-function shared-memory limit is raised
to the device maximum, never lowered to one shape's size."""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import build as mkbuild
from decode_megakernel_03_gb300 import mk, synth

pytestmark = pytest.mark.gpu

# one layer with 2048-wide rows: at batch 2 it runs the generic batch-2 kernel,
# as the tiny shape does, with a larger staging area
WIDE = synth.ModelShape("wide", 1, 2048, 16, 4, 64, 4096, 4096, tied=False, rope_theta=10000.0)


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mkbuild.build()


def _handle(shape, batch, cap, ctx):
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=0, device=dev)
    kc, vc = synth.make_kv(shape, batch, cap, ctx, seed=1, device=dev)
    dec = mk.Decoder(shape, w, kc, vc, batch)
    logits = torch.empty((batch, shape.vocab), dtype=torch.float32, device=dev)
    return dec, w, kc, vc, logits


def test_smaller_shape_does_not_lower_a_larger_handles_limit():
    big, _, _, _, lbig = _handle(WIDE, 2, 96, (40, 60))
    big.step([5, 9], [40, 60], lbig)
    assert big.status() == mk.MK_OK, big.last_error()
    first = lbig.cpu().numpy().copy()
    # a second handle of a smaller shape on the same kernel function
    small, w, kc, vc, lsmall = _handle(synth.TINY, 2, 96, (30, 31))
    small.step([1, 2], [30, 31], lsmall)
    assert small.status() == mk.MK_OK, small.last_error()
    big.step([5, 9], [40, 60], lbig)
    assert big.status() == mk.MK_OK, big.last_error()
    # the allocation-free call of the smaller shape, then the larger handle again
    rc, msg = mk.decode_step_noalloc(synth.TINY, w, kc, vc, 2, [1, 2], [30, 31], lsmall)
    assert rc == mk.MK_OK, msg
    big.step([5, 9], [40, 60], lbig)
    assert big.status() == mk.MK_OK, big.last_error()
    # the same step (same tokens, positions and cache rows) gives the same logits
    np.testing.assert_array_equal(lbig.cpu().numpy(), first)
    small.close()
    big.close()
