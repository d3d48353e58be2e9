"""Prefill as interpreter steps (mk_prefill): a prompt is written into the KV
cache in chunks of `batch` tokens, each chunk one launch whose batch rows are
the chunk's consecutive tokens of one sequence (tensor-core GEMMs over the
chunk, causal attention inside it). Checked against the oracle's full causal
forward of the same tokens: every cache row within one bf16 ulp, the logits
after the last prompt token within the parity bounds, and decoding that
continues from the prefilled cache."""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import mk, synth
from oracle import oracle as O
from tests.parity_util import KV_ATOL, KV_RTOL, Tally, bf16_bits, bits_to_f64, compare_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _check_cache(kc, vc, kf, vf, n):
    """Layer 0's rows (computed from exact embeddings: nothing compounds) within
    one bf16 ulp of the oracle's. Every layer's rows, computed from keys the
    GPU wrote for the earlier tokens, within the per-step bounds the logits
    are held to (relative L2 <= 1e-2 per row, max-abs <= 5e-2): these rows
    are intermediate activations of the whole sequence, and their rounding
    compounds through the layers. Returns the worst row rel-L2."""
    worst = 0.0
    for l in range(len(kc)):
        for got, want in ((kc[l], kf[l]), (vc[l], vf[l])):
            g = bits_to_f64(bf16_bits(got[0, :, :n]))
            o = bits_to_f64(want)
            if l == 0:
                np.testing.assert_allclose(g, o, rtol=KV_RTOL, atol=KV_ATOL)
            rel = np.linalg.norm(g - o, axis=-1) / np.maximum(np.linalg.norm(o, axis=-1), 1e-30)
            worst = max(worst, float(rel.max()))
            assert rel.max() <= 1e-2, (l, float(rel.max()))
            assert np.max(np.abs(g - o)) <= 5e-2, (l, float(np.max(np.abs(g - o))))
    return worst


@pytest.mark.parametrize("name,batch,n_prompt", [("tiny", 8, 64), ("tiny", 8, 20), ("tiny", 4, 13),
                                                 ("llama1b", 8, 24)])
def test_prefill_matches_full_forward(name, batch, n_prompt):
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    cap = 128 if name == "tiny" else 64
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=wl.weight_seed, device=dev)
    model = O.Model(shape.as_dict(), synth.oracle_weights(w))
    prompt = [int(t) for t in synth.make_tokens(shape.vocab, n_prompt, seed=21)]
    full, kf, vf = model.forward_full(np.array(prompt), want_kv=True)
    kc, vc = synth.empty_kv(shape, batch, cap, device=dev)
    dec = mk.Decoder(shape, w, kc, vc, batch)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
    dec.prefill(prompt, 0, logits)
    assert dec.status() == mk.MK_OK, dec.last_error()
    worst_row = _check_cache(kc, vc, kf, vf, n_prompt)
    tally = Tally()
    tally.add(compare_logits(logits.cpu().numpy().astype(np.float64)[None], full[-1:]))
    print(name, batch, n_prompt, tally.check(), "worst cache row rel-L2", worst_row)
    dec.close()


def test_chunked_prefill_then_decode():
    """Two prefill calls (16 tokens, then 9 more from position 16) equal one
    full forward of the 25 tokens; a batch-1 handle on the same cache then
    decodes 8 teacher-forced tokens from position 25, matching the oracle's
    forward of the whole sequence at every step."""
    wl = synth.WORKLOADS["tiny"]
    shape, cap = wl.shape, 128
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=wl.weight_seed, device=dev)
    model = O.Model(shape.as_dict(), synth.oracle_weights(w))
    seq = [int(t) for t in synth.make_tokens(shape.vocab, 33, seed=22)]
    full, kf, vf = model.forward_full(np.array(seq), want_kv=True)
    kc, vc = synth.empty_kv(shape, 8, cap, device=dev)
    pre = mk.Decoder(shape, w, kc, vc, 8)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
    pre.prefill(seq[:16], 0, logits)
    pre.prefill(seq[16:25], 16, logits)
    assert pre.status() == mk.MK_OK, pre.last_error()
    tally = Tally()
    tally.add(compare_logits(logits.cpu().numpy().astype(np.float64)[None], full[24:25]))
    _check_cache(kc, vc, [k[:, :25] for k in kf], [v[:, :25] for v in vf], 25)
    pre.close()
    # decode on sequence 0's cache (a contiguous view) with a batch-1 handle
    k1 = [t[0:1] for t in kc]
    v1 = [t[0:1] for t in vc]
    dec = mk.Decoder(shape, w, k1, v1, 1)
    lg = torch.empty((1, shape.vocab), dtype=torch.float32, device=dev)
    for t in range(25, 33):
        dec.step([seq[t]], [t], lg)
        assert dec.status() == mk.MK_OK, dec.last_error()
        tally.add(compare_logits(lg.cpu().numpy().astype(np.float64), full[t:t + 1]))
    _check_cache(kc, vc, kf, vf, 33)
    print("chunked prefill + decode", tally.check())
    dec.close()


def test_prefill_rejects_bad_arguments():
    shape = synth.TINY
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=0, device=dev)
    kc, vc = synth.empty_kv(shape, 8, 64, device=dev)
    dec = mk.Decoder(shape, w, kc, vc, 8)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
    for toks, start in (([1] * 65, 0), ([1] * 8, 57), ([shape.vocab], 0), ([], 0)):
        with pytest.raises(mk.MkError) as e:
            dec.prefill(toks, start, logits)
        assert e.value.code == mk.MK_ERR_INVALID
    dec.close()
