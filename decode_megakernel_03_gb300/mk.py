"""Thin ctypes binding of libmk.so (include/mk.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; this module
turns torch tensors into device pointers and Python lists into host arrays.
PyTorch is used for device memory and streams only. There is no fallback: if
libmk.so is missing or fails to load, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmk.so")

MK_OK, MK_ERR_INVALID, MK_ERR_CUDA, MK_ERR_TIMEOUT, MK_ERR_OOM = 0, 1, 2, 3, 4
OPS = {1: "QKV", 2: "ATTN", 3: "RED", 4: "OPROJ", 5: "GATEUP", 6: "DOWN", 7: "LMHEAD"}
OP_QKV, OP_ATTN, OP_RED, OP_OPROJ, OP_GATEUP, OP_DOWN, OP_LMHEAD = range(1, 8)

# exported entry points (the C-ABI surface declared in include/mk.h)
EXPORTS = ("mk_create", "mk_decode_step", "mk_decode_step_multilaunch", "mk_get_status",
           "mk_destroy", "mk_last_error", "mk_read_counters", "mk_set_timeout",
           "mk_debug_inject_unsatisfiable_wait", "mk_set_trace", "mk_schedule_build",
           "mk_decode_step_noalloc", "mk_debug_use_generic_kernel", "mk_decode_greedy",
           "mk_create_paged", "mk_decode_step_paged", "mk_decode_greedy_persistent",
           "mk_debug_permute_queues", "mk_set_dynamic", "mk_schedule_build_dynamic",
           "mk_schedule_build_steps", "mk_prefill")

MAX_STEPS_PER_LAUNCH = 32  # MK_MAX_STEPS_PER_LAUNCH

MAX_GREEDY_STEPS = 1024  # MK_MAX_GREEDY_STEPS


class MkError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"mk error {code}: {msg}")
        self.code = code


class MkConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("tied_embeddings", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("batch", ctypes.c_int), ("kv_capacity", ctypes.c_int)]


_vpp = ctypes.POINTER(ctypes.c_void_p)


class MkWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("final_norm", ctypes.c_void_p), ("attn_norm", _vpp), ("wq", _vpp), ("wk", _vpp),
                ("wv", _vpp), ("wo", _vpp), ("mlp_norm", _vpp), ("wgate", _vpp), ("wup", _vpp),
                ("wdown", _vpp)]


class MkInstr(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int16), ("layer", ctypes.c_int16), ("a0", ctypes.c_int32),
                ("a1", ctypes.c_int32), ("a2", ctypes.c_int32), ("wait_ctr", ctypes.c_int32),
                ("wait_target", ctypes.c_int32), ("sig_ctr", ctypes.c_int32),
                ("sig_amount", ctypes.c_int32)]


INSTR_DTYPE = np.dtype([("op", "<i2"), ("layer", "<i2"), ("a0", "<i4"), ("a1", "<i4"),
                        ("a2", "<i4"), ("wait_ctr", "<i4"), ("wait_target", "<i4"),
                        ("sig_ctr", "<i4"), ("sig_amount", "<i4")])
TRACE_DTYPE = np.dtype([("sm", "<u4"), ("index", "<u4"), ("op", "<i4"), ("layer", "<i4"),
                        ("t_start", "<u8"), ("t_ready", "<u8"), ("t_end", "<u8"),
                        ("t_stored", "<u8"), ("res_wait_ns", "<u4"), ("stage_ns", "<u4"),
                        ("t_issue_first", "<u8"), ("t_issue_last", "<u8"),
                        ("page_wait_ns", "<u4"), ("reserved", "<u4")])

_lib = None


def lib():
    """Loads libmk.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run decode_megakernel_03_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
        L.mk_create.argtypes = [ctypes.POINTER(MkConfig), ctypes.POINTER(MkWeights), _vpp, _vpp,
                                ctypes.POINTER(vp)]
        L.mk_decode_step.argtypes = [vp, i32p, i32p, vp, vp]
        L.mk_decode_step_multilaunch.argtypes = [vp, i32p, i32p, vp, vp, ctypes.c_int]
        L.mk_decode_greedy.argtypes = [vp, i32p, i32p, ctypes.c_int, vp, vp, vp]
        L.mk_create_paged.argtypes = [ctypes.POINTER(MkConfig), ctypes.POINTER(MkWeights), _vpp,
                                      _vpp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp)]
        L.mk_decode_step_paged.argtypes = [vp, i32p, i32p, i32p, vp, vp]
        L.mk_decode_greedy_persistent.argtypes = [vp, i32p, i32p, ctypes.c_int, vp, vp, vp]
        L.mk_get_status.argtypes = [vp, vp]
        L.mk_destroy.argtypes = [vp]
        L.mk_last_error.argtypes = [vp]
        L.mk_last_error.restype = ctypes.c_char_p
        L.mk_read_counters.argtypes = [vp, i32p, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        L.mk_set_timeout.argtypes = [vp, ctypes.c_uint64]
        L.mk_debug_inject_unsatisfiable_wait.argtypes = [vp, ctypes.c_int]
        L.mk_debug_use_generic_kernel.argtypes = [vp, ctypes.c_int]
        L.mk_debug_permute_queues.argtypes = [vp, ctypes.c_uint32]
        L.mk_set_dynamic.argtypes = [vp, ctypes.c_int]
        L.mk_prefill.argtypes = [vp, i32p, ctypes.c_int, ctypes.c_int, vp, vp]
        L.mk_schedule_build_steps.argtypes = [ctypes.POINTER(MkConfig), ctypes.c_int, i32p,
                                              ctypes.c_int, ctypes.POINTER(MkInstr),
                                              ctypes.c_int, ctypes.POINTER(ctypes.c_int), i32p,
                                              i32p, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        L.mk_schedule_build_dynamic.argtypes = [ctypes.POINTER(MkConfig), ctypes.c_int, i32p,
                                                ctypes.c_int, ctypes.POINTER(MkInstr),
                                                ctypes.c_int, ctypes.POINTER(ctypes.c_int), i32p,
                                                i32p, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        L.mk_set_trace.argtypes = [vp, vp, ctypes.c_int]
        L.mk_schedule_build.argtypes = [ctypes.POINTER(MkConfig), ctypes.c_int, i32p,
                                        ctypes.POINTER(MkInstr), ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int), i32p, i32p, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int)]
        L.mk_decode_step_noalloc.argtypes = [ctypes.POINTER(MkConfig), ctypes.POINTER(MkWeights),
                                             _vpp, _vpp, i32p, i32p, vp, vp, ctypes.c_char_p,
                                             ctypes.c_size_t]
        _lib = L
    return _lib


def _err(h) -> str:
    s = lib().mk_last_error(h)
    return s.decode() if s else ""


def _check(rc: int, h=None):
    if rc != MK_OK:
        raise MkError(rc, _err(h))


def make_config(shape, batch: int, capacity: int) -> MkConfig:
    return MkConfig(shape.n_layers, shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                    shape.ffn, shape.vocab, int(bool(shape.tied)), float(shape.rms_eps),
                    float(shape.rope_theta), int(batch), int(capacity))


def _i32(vals, n: int | None = None):
    """A host int32 array of vals; n: the length the library will read."""
    if n is not None and len(vals) != n:
        raise MkError(MK_ERR_INVALID, f"expected {n} values, got {len(vals)}")
    a = (ctypes.c_int32 * len(vals))(*[int(v) for v in vals])
    return a


def _dev(t, n: int, dtype: str, what: str) -> ctypes.c_void_p:
    """The device pointer of tensor t after checking that the library may
    write n elements of dtype there (it cannot check that itself)."""
    if not t.is_cuda or str(t.dtype) != "torch." + dtype or not t.is_contiguous():
        raise MkError(MK_ERR_INVALID, f"{what} must be a contiguous CUDA {dtype} tensor")
    if t.numel() < n:
        raise MkError(MK_ERR_INVALID, f"{what} holds {t.numel()} elements, {n} are written")
    return ctypes.c_void_p(t.data_ptr())


DYN_LMHEAD = 1  # MK_DYN_LMHEAD


def schedule(shape, batch: int, capacity: int, n_sm: int, positions, dyn: int = 0):
    """Host-only schedule: (instrs structured array, sm_offsets, counter targets).
    dyn: MK_DYN_* flags (0: the static plan)."""
    cfg = make_config(shape, batch, capacity)
    n_instr, n_ctr = ctypes.c_int(0), ctypes.c_int(0)
    pos = _i32(positions)
    rc = lib().mk_schedule_build_dynamic(ctypes.byref(cfg), n_sm, pos, int(dyn), None, 0,
                                         ctypes.byref(n_instr), None, None, 0,
                                         ctypes.byref(n_ctr))
    _check(rc)
    instrs = (MkInstr * n_instr.value)()
    offs = (ctypes.c_int32 * (n_sm + 1))()
    tg = (ctypes.c_int32 * n_ctr.value)()
    rc = lib().mk_schedule_build_dynamic(ctypes.byref(cfg), n_sm, pos, int(dyn), instrs,
                                         n_instr.value, ctypes.byref(n_instr), offs, tg,
                                         n_ctr.value, ctypes.byref(n_ctr))
    _check(rc)
    arr = np.frombuffer(bytes(instrs), dtype=INSTR_DTYPE).copy()
    return arr, np.array(offs, dtype=np.int64), np.array(tg, dtype=np.int64)


def schedule_steps(shape, batch: int, capacity: int, n_sm: int, positions, n_steps: int):
    """Host-only schedule of n_steps greedy steps in one launch (the plan of
    mk_decode_greedy_persistent): (instrs, sm_offsets, counter targets)."""
    cfg = make_config(shape, batch, capacity)
    n_instr, n_ctr = ctypes.c_int(0), ctypes.c_int(0)
    pos = _i32(positions)
    rc = lib().mk_schedule_build_steps(ctypes.byref(cfg), n_sm, pos, int(n_steps), None, 0,
                                       ctypes.byref(n_instr), None, None, 0, ctypes.byref(n_ctr))
    _check(rc)
    instrs = (MkInstr * n_instr.value)()
    offs = (ctypes.c_int32 * (n_sm + 1))()
    tg = (ctypes.c_int32 * n_ctr.value)()
    rc = lib().mk_schedule_build_steps(ctypes.byref(cfg), n_sm, pos, int(n_steps), instrs,
                                       n_instr.value, ctypes.byref(n_instr), offs, tg,
                                       n_ctr.value, ctypes.byref(n_ctr))
    _check(rc)
    arr = np.frombuffer(bytes(instrs), dtype=INSTR_DTYPE).copy()
    return arr, np.array(offs, dtype=np.int64), np.array(tg, dtype=np.int64)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _model_structs(shape, weights: dict, k_cache: list, v_cache: list, batch: int):
    """ctypes mk_config / mk_weights / cache pointer arrays for torch tensors;
    the last element keeps the host arrays alive."""
    L = shape.n_layers
    arrs = {}
    for name in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown"):
        arrs[name] = (ctypes.c_void_p * L)(*[t.data_ptr() for t in weights[name]])
    lm = weights.get("lm_head")
    w = MkWeights(weights["embed"].data_ptr(), lm.data_ptr() if lm is not None else None,
                  weights["final_norm"].data_ptr(),
                  *[ctypes.cast(arrs[n], _vpp) for n in ("attn_norm", "wq", "wk", "wv", "wo",
                                                         "mlp_norm", "wgate", "wup", "wdown")])
    kc = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_cache])
    vc = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_cache])
    cfg = make_config(shape, batch, int(k_cache[0].shape[2]))
    return cfg, w, kc, vc, (arrs, weights, k_cache, v_cache)


def decode_step_noalloc(shape, weights: dict, k_cache: list, v_cache: list, batch: int, tokens,
                        positions, logits, stream=None):
    """mk_decode_step_noalloc: one decode step with no handle and no device
    allocation (scratch in the library's static device array). Synchronous.
    Returns (status code, message)."""
    cfg, w, kc, vc, keep = _model_structs(shape, weights, k_cache, v_cache, batch)
    msg = ctypes.create_string_buffer(512)
    rc = lib().mk_decode_step_noalloc(ctypes.byref(cfg), ctypes.byref(w), ctypes.cast(kc, _vpp),
                                      ctypes.cast(vc, _vpp), _i32(tokens, batch),
                                      _i32(positions, batch),
                                      _dev(logits, batch * shape.vocab, "float32", "logits"),
                                      _stream_ptr(stream), msg, len(msg))
    del keep
    return rc, msg.value.decode()


class Decoder:
    """One handle: a model (weights on the device), a batch and its KV cache.

    weights: dict of torch bf16 CUDA tensors as produced by synth.make_weights
    (per-layer lists for the layer matrices); k_cache / v_cache: lists of
    [B][nkv][S][D] bf16 CUDA tensors, updated in place by every step.
    """

    def __init__(self, shape, weights: dict, k_cache: list, v_cache: list, batch: int,
                 paged=None):
        """paged = (block_size, n_blocks, kv_capacity): k_cache / v_cache are
        block pools [n_blocks][nkv][block_size][D] (mk_create_paged), stepped
        with step_paged."""
        self.shape = shape
        self.batch = batch
        self.capacity = int(k_cache[0].shape[2]) if paged is None else int(paged[2])
        # block-table entries per sequence of a paged handle
        self.max_blocks = 0 if paged is None else -(-self.capacity // int(paged[0]))
        L = shape.n_layers
        self._keep = (weights, k_cache, v_cache)
        arrs = {}
        for name in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown"):
            arrs[name] = (ctypes.c_void_p * L)(*[t.data_ptr() for t in weights[name]])
        self._arrs = arrs
        lm = weights.get("lm_head")
        self._w = MkWeights(weights["embed"].data_ptr(), lm.data_ptr() if lm is not None else None,
                            weights["final_norm"].data_ptr(),
                            *[ctypes.cast(arrs[n], _vpp) for n in ("attn_norm", "wq", "wk", "wv",
                                                                   "wo", "mlp_norm", "wgate",
                                                                   "wup", "wdown")])
        self._kc = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_cache])
        self._vc = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_cache])
        self.cfg = make_config(shape, batch, self.capacity)
        h = ctypes.c_void_p()
        if paged is None:
            rc = lib().mk_create(ctypes.byref(self.cfg), ctypes.byref(self._w),
                                 ctypes.cast(self._kc, _vpp), ctypes.cast(self._vc, _vpp),
                                 ctypes.byref(h))
        else:
            rc = lib().mk_create_paged(ctypes.byref(self.cfg), ctypes.byref(self._w),
                                       ctypes.cast(self._kc, _vpp), ctypes.cast(self._vc, _vpp),
                                       int(paged[0]), int(paged[1]), ctypes.byref(h))
        _check(rc, None)
        self.h = h

    # -- decode ----------------------------------------------------------
    def _logits(self, logits, rows: int | None = None) -> ctypes.c_void_p:
        n = (self.batch if rows is None else rows) * self.shape.vocab
        return _dev(logits, n, "float32", "logits")

    def _tokens_out(self, t, n_steps: int, most: int) -> ctypes.c_void_p:
        # a step count out of range is refused by the library before it
        # writes anything, so only a valid count sizes the check
        n = n_steps * self.batch if 1 <= n_steps <= most else 0
        return _dev(t, n, "int32", "tokens_out")

    def step(self, tokens, positions, logits, stream=None) -> int:
        rc = lib().mk_decode_step(self.h, _i32(tokens, self.batch), _i32(positions, self.batch),
                                  self._logits(logits), _stream_ptr(stream))
        _check(rc, self.h)
        return rc

    def prefill(self, tokens, start_pos: int, logits, stream=None) -> int:
        """mk_prefill: the prompt into sequence 0 of the cache, in chunks of
        `batch` tokens; logits (device fp32 [vocab]) receives the logits after
        the last prompt token."""
        rc = lib().mk_prefill(self.h, _i32(tokens), len(tokens), int(start_pos),
                              self._logits(logits, 1), _stream_ptr(stream))
        _check(rc, self.h)
        return rc

    def step_paged(self, tokens, positions, block_table, logits, stream=None) -> int:
        """mk_decode_step_paged; block_table: int32 numpy array
        [batch][ceil(kv_capacity / block_size)] on the host."""
        tbl = np.ascontiguousarray(block_table, dtype=np.int32)
        if self.max_blocks and tbl.size != self.batch * self.max_blocks:
            raise MkError(MK_ERR_INVALID, f"block_table must hold batch x {self.max_blocks} entries")
        rc = lib().mk_decode_step_paged(self.h, _i32(tokens, self.batch),
                                        _i32(positions, self.batch),
                                        tbl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                        self._logits(logits), _stream_ptr(stream))
        _check(rc, self.h)
        return rc

    def decode_greedy(self, tokens, positions, n_steps: int, tokens_out, logits,
                      stream=None) -> int:
        """mk_decode_greedy: n_steps greedy steps, the tokens fed back on the
        device; tokens_out is a device int32 tensor of n_steps * batch."""
        rc = lib().mk_decode_greedy(self.h, _i32(tokens, self.batch), _i32(positions, self.batch),
                                    int(n_steps), self._tokens_out(tokens_out, n_steps,
                                                                   MAX_GREEDY_STEPS),
                                    self._logits(logits), _stream_ptr(stream))
        _check(rc, self.h)
        return rc

    def decode_greedy_persistent(self, tokens, positions, n_steps: int, tokens_out, logits,
                                 stream=None) -> int:
        """mk_decode_greedy_persistent: n_steps greedy steps in one launch."""
        rc = lib().mk_decode_greedy_persistent(
            self.h, _i32(tokens, self.batch), _i32(positions, self.batch), int(n_steps),
            self._tokens_out(tokens_out, n_steps, MAX_STEPS_PER_LAUNCH), self._logits(logits),
            _stream_ptr(stream))
        _check(rc, self.h)
        return rc

    def step_multilaunch(self, tokens, positions, logits, stream=None, graph: bool = False) -> int:
        rc = lib().mk_decode_step_multilaunch(self.h, _i32(tokens, self.batch),
                                              _i32(positions, self.batch), self._logits(logits),
                                              _stream_ptr(stream), int(bool(graph)))
        _check(rc, self.h)
        return rc

    def status(self, stream=None) -> int:
        """mk_get_status: returns the code (does not raise on MK_ERR_TIMEOUT)."""
        return lib().mk_get_status(self.h, _stream_ptr(stream))

    def counters(self) -> np.ndarray:
        n = ctypes.c_int(0)
        lib().mk_read_counters(self.h, None, 0, ctypes.byref(n))
        buf = (ctypes.c_int32 * n.value)()
        _check(lib().mk_read_counters(self.h, buf, n.value, ctypes.byref(n)), self.h)
        return np.array(buf, dtype=np.int64)

    def set_timeout(self, ns: int):
        _check(lib().mk_set_timeout(self.h, int(ns)), self.h)

    def use_generic_kernel(self, enable: bool):
        """Test hook: launch the instantiation that reads the head shape at run time."""
        _check(lib().mk_debug_use_generic_kernel(self.h, int(bool(enable))), self.h)

    def set_dynamic(self, flags: int):
        """mk_set_dynamic: MK_DYN_* flags (0: the static plan)."""
        _check(lib().mk_set_dynamic(self.h, int(flags)), self.h)

    def permute_queues(self, seed: int):
        """Test hook: hand the per-SM queues to the CTAs in a seeded order."""
        _check(lib().mk_debug_permute_queues(self.h, int(seed)), self.h)

    def inject_unsatisfiable_wait(self, enable: bool):
        _check(lib().mk_debug_inject_unsatisfiable_wait(self.h, int(bool(enable))), self.h)

    def set_trace(self, buf=None):
        """buf: a torch uint8 CUDA tensor of n * TRACE_DTYPE.itemsize bytes, or
        None to disable."""
        if buf is None:
            _check(lib().mk_set_trace(self.h, None, 0), self.h)
        else:
            _check(lib().mk_set_trace(self.h, ctypes.c_void_p(buf.data_ptr()),
                                      buf.numel() // TRACE_DTYPE.itemsize), self.h)

    def last_error(self) -> str:
        return _err(self.h)

    def close(self):
        if getattr(self, "h", None):
            lib().mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
