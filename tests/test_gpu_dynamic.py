"""Dynamic work distribution (mk_set_dynamic, MK_DYN_LMHEAD): the LM head's
row blocks taken at run time from a per-step ticket counter by whichever SM
reaches them. The results must equal the static plan's bit for bit (a row's
arithmetic does not depend on the SM that runs it), every counter must reach
its target, and the ticket counter must have handed out every block once
(plus the one failed take of each SM)."""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import mk, synth
from tests.parity_util import Pair, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


@pytest.mark.parametrize("name", ["tiny", "llama1b", "llama1b_b8"])
def test_dynamic_lm_head_equals_static(name):
    wl = synth.WORKLOADS[name]
    ctx = (50,) if name == "tiny" else wl.ctx
    cap = 128 if name == "tiny" else wl.capacity
    toks = synth.step_tokens(wl)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    out = {}
    for dyn in (0, mk.DYN_LMHEAD):
        pair = Pair(wl.shape, wl.batch, cap, ctx=ctx)
        pair.dec.set_dynamic(dyn)
        res = []
        for s in range(3):
            tok = [int(t) for t in toks[s][:wl.batch]]
            pos = [c + s for c in ctx]
            res.append(pair.gpu_step(tok, pos))
        out[dyn] = (np.stack(res), [bf16_bits(t) for t in pair.kc + pair.vc])
        ins, off, tg = mk.schedule(wl.shape, wl.batch, cap, n_sm, pos, dyn=dyn)
        got = pair.dec.counters()
        if dyn:
            lm = ins[ins["op"] == mk.OP_LMHEAD]
            tk = int(lm["a2"][0]) - 1
            n_tickets = -(-wl.shape.vocab // int(lm["a0"][0]))
            assert got[tk] == n_tickets + n_sm
            got = got.copy()
            got[tk] = 0
        np.testing.assert_array_equal(got, tg)
        pair.close()
    np.testing.assert_array_equal(out[0][0], out[mk.DYN_LMHEAD][0])
    for a, b in zip(out[0][1], out[mk.DYN_LMHEAD][1]):
        np.testing.assert_array_equal(a, b)


def test_dynamic_flag_leaves_greedy_and_paged_steps_static():
    """Greedy decode and paged steps run the feature kernels, built without
    dynamic distribution: a handle with the flag set still decodes them with
    the static plan, and gives the same tokens as without the flag."""
    wl = synth.WORKLOADS["llama1b"]
    toks = {}
    for dyn in (0, mk.DYN_LMHEAD):
        pair = Pair(wl.shape, 1, wl.capacity, ctx=wl.ctx)
        pair.dec.set_dynamic(dyn)
        out = torch.empty(8, dtype=torch.int32, device="cuda")
        pair.dec.decode_greedy_persistent([17], [512], 8, out, pair.logits)
        assert pair.dec.status() == mk.MK_OK, pair.dec.last_error()
        toks[dyn] = (out.cpu().numpy().copy(), pair.logits.cpu().numpy().copy())
        pair.close()
    np.testing.assert_array_equal(toks[0][0], toks[mk.DYN_LMHEAD][0])
    np.testing.assert_array_equal(toks[0][1], toks[mk.DYN_LMHEAD][1])


def test_dynamic_flag_rejected_without_a_build():
    """A shape without a dynamic instantiation refuses the flag."""
    shape = synth.ModelShape("d128g2", 1, 512, 4, 2, 128, 1024, 4096, tied=False)
    pair = Pair(shape, 2, 64, ctx=(10, 20))
    with pytest.raises(mk.MkError) as e:
        pair.dec.set_dynamic(mk.DYN_LMHEAD)
    assert e.value.code == mk.MK_ERR_INVALID
    pair.dec.set_dynamic(0)
    pair.close()
