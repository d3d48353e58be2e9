"""The C-ABI library: it loads without a GPU, exports every entry point that
include/mk.h declares, and rejects bad arguments on the host before touching
CUDA. No compute call is made here."""
import ctypes
import os
import re

import pytest

from decode_megakernel_03_gb300 import build as mkbuild
from decode_megakernel_03_gb300 import mk, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mkbuild.build()
    return mk.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared()
    for n in ("mk_create", "mk_decode_step", "mk_destroy"):
        assert n in names
    assert set(names) == set(mk.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_create_rejects_bad_arguments_on_host(L):
    h = ctypes.c_void_p(123)
    assert L.mk_create(None, None, None, None, ctypes.byref(h)) == mk.MK_ERR_INVALID
    assert h.value is None
    assert b"NULL" in L.mk_last_error(None)
    cfg = mk.make_config(synth.TINY, 1, 128)
    cfg.head_dim = 96
    assert L.mk_create(ctypes.byref(cfg), None, None, None, ctypes.byref(h)) == mk.MK_ERR_INVALID
    assert b"head_dim" in L.mk_last_error(None)
    cfg = mk.make_config(synth.TINY, 3, 128)
    assert L.mk_create(ctypes.byref(cfg), None, None, None, ctypes.byref(h)) == mk.MK_ERR_INVALID
    assert b"batch" in L.mk_last_error(None)
    cfg = mk.make_config(synth.TINY, 1, 128)
    w = mk.MkWeights()
    assert L.mk_create(ctypes.byref(cfg), ctypes.byref(w), None, None,
                       ctypes.byref(h)) == mk.MK_ERR_INVALID


def test_null_handle_is_invalid(L):
    assert L.mk_decode_step(None, None, None, None, None) == mk.MK_ERR_INVALID
    assert L.mk_get_status(None, None) == mk.MK_ERR_INVALID
    assert L.mk_destroy(None) == mk.MK_OK


def test_schedule_rejects_out_of_range_positions(L):
    with pytest.raises(mk.MkError) as e:
        mk.schedule(synth.TINY, 1, 128, 8, [128])
    assert e.value.code == mk.MK_ERR_INVALID
    with pytest.raises(mk.MkError):
        mk.schedule(synth.TINY, 1, 128, 8, [-1])


@pytest.mark.parametrize("field,value", [("hidden", 300), ("ffn", 1000), ("n_kv_heads", 3),
                                         ("n_heads", 40), ("hidden", 8192)])
def test_unsupported_shapes(L, field, value):
    cfg = mk.make_config(synth.TINY, 1, 128)
    setattr(cfg, field, value)
    n = ctypes.c_int()
    pos = (ctypes.c_int32 * 1)(0)
    rc = L.mk_schedule_build(ctypes.byref(cfg), 4, pos, None, 0, ctypes.byref(n), None, None, 0,
                             ctypes.byref(n))
    assert rc == mk.MK_ERR_INVALID


def test_binding_checks_what_the_library_cannot():
    """The library reads B host token ids and positions and writes B x vocab
    logits through bare pointers; the binding refuses lists of another length
    and output tensors that are not contiguous CUDA tensors of the right type
    and size, before anything is passed on."""
    import torch

    with pytest.raises(mk.MkError) as e:
        mk._i32([1, 2], 3)
    assert e.value.code == mk.MK_ERR_INVALID
    assert list(mk._i32([4, 5, 6], 3)) == [4, 5, 6]
    for t, n, dt in ((torch.empty(8), 8, "float32"),                     # host memory
                     (torch.empty(8, dtype=torch.int32), 8, "float32")):  # wrong type
        with pytest.raises(mk.MkError) as e:
            mk._dev(t, n, dt, "logits")
        assert e.value.code == mk.MK_ERR_INVALID
