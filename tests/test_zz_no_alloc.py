"""mk_decode_step_noalloc, the decode step for callers that may not allocate
device memory (code inside a pool or arena that owns every device byte,
plugins whose host forbids allocations after start-up): its scratch lives in
the library's static device array. Called through the C ABI, two steps in a
row, it must agree with mk_decode_step on the same inputs, within the
tolerances the parity tests use. This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import build as mkbuild
from decode_megakernel_03_gb300 import mk, synth
from tests.parity_util import KV_ATOL, KV_RTOL, Tally, bf16_bits, bits_to_f64, compare_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mkbuild.build()


def _inputs(shape, batch, cap, ctx):
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=0, device=dev)
    kc, vc = synth.make_kv(shape, batch, cap, ctx, seed=1, device=dev)
    return w, kc, vc


@pytest.mark.parametrize("name,batch,cap,ctx", [
    ("tiny", 1, 128, (40,)),
    ("llama1b", 1, 640, (512,)),
    ("tiny", 2, 160, (17, 90)),
])
def test_noalloc_matches_handle_path_two_calls(name, batch, cap, ctx):
    shape = synth.WORKLOADS[name].shape
    w, kc_a, vc_a = _inputs(shape, batch, cap, ctx)
    _, kc_b, vc_b = _inputs(shape, batch, cap, ctx)  # an identical second copy of the caches
    dec = mk.Decoder(shape, w, kc_a, vc_a, batch)
    la = torch.empty((batch, shape.vocab), dtype=torch.float32, device="cuda")
    lb = torch.empty_like(la)
    tally = Tally()
    toks = synth.step_tokens(synth.WORKLOADS[name])
    for s in range(2):
        tok = [(int(toks[s, b % toks.shape[1]]) + b) % shape.vocab for b in range(batch)]
        pos = [c + s for c in ctx]
        dec.step(tok, pos, la)
        assert dec.status() == mk.MK_OK, dec.last_error()
        rc, msg = mk.decode_step_noalloc(shape, w, kc_b, vc_b, batch, tok, pos, lb)
        assert rc == mk.MK_OK, msg
        tally.add(compare_logits(lb.cpu().numpy().astype(np.float64),
                                 la.cpu().numpy().astype(np.float64)))
    tally.check()
    for a, b in zip(kc_a + vc_a, kc_b + vc_b):
        np.testing.assert_allclose(bits_to_f64(bf16_bits(b)), bits_to_f64(bf16_bits(a)),
                                   rtol=KV_RTOL, atol=KV_ATOL)
    dec.close()


def test_noalloc_rejects_scratch_beyond_its_array():
    shape = synth.TINY
    cap = 65536  # the RoPE table alone would need 16.8 MB of the 16 MiB array
    w, kc, vc = _inputs(shape, 1, cap, (10,))
    logits = torch.empty((1, shape.vocab), dtype=torch.float32, device="cuda")
    rc, msg = mk.decode_step_noalloc(shape, w, kc, vc, 1, [3], [10], logits)
    assert rc == mk.MK_ERR_INVALID
    assert "needs" in msg and "static array" in msg
