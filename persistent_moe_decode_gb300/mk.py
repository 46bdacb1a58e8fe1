"""Python binding of the C ABI in include/mk.h (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the decode step: the step runs in the CUDA kernels of libmk.so.
The library is loaded on first use; if it has not been built the binding
raises (there is no fallback path).
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmk.so")
_lock = threading.Lock()
_lib = None

MK_OK = 0
MK_ERR_BAD_CONFIG = -1
MK_ERR_OOM = -2
MK_ERR_BAD_PAGE = -3
MK_ERR_BATCH_TOO_LARGE = -4
MK_ERR_NOT_SCHEDULED = -5
MK_ERR_TIMEOUT = -6
MK_ERR_CUDA = -7
MK_ERR_BAD_ARG = -8
MK_ERR_DEVICE = -9

MK_WAVES_DEFAULT, MK_WAVES_ATTN_FIRST, MK_WAVES_INTERLEAVED = 0, 1, 2
MK_EXPERTS_BF16, MK_EXPERTS_FP8_E4M3 = 0, 1
(MK_SCRATCH_H, MK_SCRATCH_X, MK_SCRATCH_QKV, MK_SCRATCH_ATTN, MK_SCRATCH_ROUTER,
 MK_SCRATCH_OPROJ, MK_SCRATCH_MOE) = range(7)
MK_DEBUG_ROUTE_GROUPS, MK_DEBUG_PAGE_GATHER, MK_DEBUG_NEW_SLOT = range(3)

# every symbol include/mk.h declares
EXPORTS = ("mk_create", "mk_schedule_step", "mk_decode_step", "mk_step_status", "mk_get_routing",
           "mk_read_scratch", "mk_plan", "mk_debug_bump_wait", "mk_device_bytes", "mk_num_sms",
           "mk_step_upload_bytes", "mk_destroy", "mk_strerror", "mk_abi_version", "mk_read_trace",
           "mk_decode_step_static", "mk_plan_step", "mk_read_debug", "mk_service_create",
           "mk_service_submit", "mk_service_run", "mk_service_wait", "mk_service_result",
           "mk_service_batch", "mk_service_destroy")


class mk_config(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("hidden", C.c_int), ("n_q_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("n_experts", C.c_int),
                ("top_k", C.c_int), ("moe_inter", C.c_int), ("vocab", C.c_int),
                ("page_size", C.c_int), ("rope_theta", C.c_double), ("rms_eps", C.c_float),
                ("max_batch", C.c_int), ("max_pages_per_seq", C.c_int), ("num_kv_pages", C.c_int),
                ("max_attn_items", C.c_int), ("wave_order", C.c_int), ("n_attn_claimers", C.c_int),
                ("n_moe_claimers", C.c_int), ("kv_split_tokens", C.c_int), ("sm_cap", C.c_int),
                ("timeout_ms", C.c_int), ("trace_records", C.c_int), ("moe_stage_depth", C.c_int),
                ("expert_format", C.c_int), ("moe_claim_rows", C.c_int)]


_VPP = C.POINTER(C.c_void_p)


class mk_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("attn_norm", _VPP), ("w_qkv", _VPP), ("w_o", _VPP), ("w_router", _VPP),
                ("w_gate", _VPP), ("w_up", _VPP), ("w_down", _VPP), ("k_pool", _VPP),
                ("v_pool", _VPP), ("s_gate", _VPP), ("s_up", _VPP), ("s_down", _VPP)]


class mk_error(C.Structure):
    _fields_ = [("code", C.c_int), ("sm", C.c_int), ("task", C.c_int), ("op", C.c_int),
                ("barrier", C.c_int), ("value", C.c_uint), ("target", C.c_uint)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class MkError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {mk_strerror(code)} ({code})")
        self.code = code


def lib():
    """Load libmk.so; raise if it is missing (no CPU fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is not built: run `python -m "
                                   "persistent_moe_decode_gb300.build` (needs nvcc)")
            L = C.CDLL(_LIB_PATH)
            vp, i32 = C.c_void_p, C.c_int
            L.mk_create.argtypes = [C.POINTER(mk_config), C.POINTER(mk_weights), C.POINTER(vp)]
            L.mk_schedule_step.argtypes = [vp, i32, vp, vp, vp, vp, vp]
            L.mk_decode_step.argtypes = [vp, vp, vp]
            L.mk_decode_step_static.argtypes = [vp, vp, vp]
            L.mk_step_status.argtypes = [vp, C.POINTER(mk_error)]
            L.mk_get_routing.argtypes = [vp, vp, vp]
            L.mk_read_scratch.argtypes = [vp, i32, i32, vp, C.c_size_t, C.POINTER(C.c_size_t)]
            L.mk_plan.argtypes = [C.POINTER(mk_config), i32, i32, vp, vp, C.POINTER(i32),
                                  C.POINTER(i32)]
            L.mk_plan_step.argtypes = [C.POINTER(mk_config), i32, i32, vp, vp, vp, vp, vp, vp, vp]
            L.mk_debug_bump_wait.argtypes = [vp, i32, i32]
            L.mk_read_trace.argtypes = [vp, vp, C.c_size_t, C.POINTER(C.c_size_t)]
            L.mk_read_debug.argtypes = [vp, i32, vp, C.c_size_t, C.POINTER(C.c_size_t)]
            L.mk_service_create.argtypes = [vp, vp, C.POINTER(vp)]
            L.mk_service_submit.argtypes = [vp, vp, i32, i32, i32, i32, C.POINTER(C.c_int64)]
            L.mk_service_run.argtypes = [vp, i32]
            L.mk_service_wait.argtypes = [vp]
            L.mk_service_result.argtypes = [vp, C.c_int64, vp, i32, C.POINTER(i32), C.POINTER(i32)]
            L.mk_service_batch.argtypes = [vp, vp, vp, vp, C.POINTER(i32)]
            L.mk_service_destroy.argtypes = [vp]
            L.mk_service_destroy.restype = None
            L.mk_device_bytes.argtypes = [vp]
            L.mk_device_bytes.restype = C.c_size_t
            L.mk_num_sms.argtypes = [vp]
            L.mk_step_upload_bytes.argtypes = [vp, i32]
            L.mk_step_upload_bytes.restype = C.c_size_t
            L.mk_destroy.argtypes = [vp]
            L.mk_destroy.restype = None
            L.mk_strerror.argtypes = [i32]
            L.mk_strerror.restype = C.c_char_p
            _lib = L
    return _lib


def _check(rc: int, where: str) -> int:
    if rc != MK_OK:
        raise MkError(rc, where)
    return rc


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _stream_ptr(stream):
    if stream is None:
        return None
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ------------------------------------------------------------- entry points

def mk_strerror(code: int) -> str:
    return lib().mk_strerror(int(code)).decode()


def mk_abi_version() -> int:
    return int(lib().mk_abi_version())


def mk_create(cfg: mk_config, weights: mk_weights):
    h = C.c_void_p()
    _check(lib().mk_create(C.byref(cfg), C.byref(weights), C.byref(h)), "mk_create")
    return h


def mk_schedule_step(h, batch: int, seq_ids, tokens, page_tables, seq_lens, stream=None) -> int:
    tok, pt, sl = _i32(tokens), _i32(page_tables), _i32(seq_lens)
    sid = _i32(seq_ids) if seq_ids is not None else None
    return _check(lib().mk_schedule_step(h, int(batch), _ptr(sid) if sid is not None else None,
                                         _ptr(tok), _ptr(pt), _ptr(sl), _stream_ptr(stream)),
                  "mk_schedule_step")


def mk_decode_step(h, logits_ptr: int, stream=None) -> int:
    return _check(lib().mk_decode_step(h, C.c_void_p(int(logits_ptr)), _stream_ptr(stream)),
                  "mk_decode_step")


def mk_decode_step_static(h, logits_ptr: int, stream=None) -> int:
    return _check(lib().mk_decode_step_static(h, C.c_void_p(int(logits_ptr)), _stream_ptr(stream)),
                  "mk_decode_step_static")


def mk_step_status(h):
    e = mk_error()
    rc = lib().mk_step_status(h, C.byref(e))
    return rc, e


def mk_get_routing(h, n_layers: int, batch: int, top_k: int):
    idx = np.empty((n_layers, batch, top_k), dtype=np.int32)
    w = np.empty((n_layers, batch, top_k), dtype=np.float32)
    _check(lib().mk_get_routing(h, _ptr(idx), _ptr(w)), "mk_get_routing")
    return idx, w


def mk_read_scratch(h, which: int, layer: int) -> bytes:
    size = C.c_size_t(0)
    _check(lib().mk_read_scratch(h, int(which), int(layer), None, 0, C.byref(size)), "mk_read_scratch")
    buf = (C.c_uint8 * size.value)()
    _check(lib().mk_read_scratch(h, int(which), int(layer), C.cast(buf, C.c_void_p), size.value, None),
           "mk_read_scratch")
    return bytes(buf)


def mk_plan(cfg: mk_config, n_sm: int, batch: int):
    n_tasks, n_bars = C.c_int(0), C.c_int(0)
    _check(lib().mk_plan(C.byref(cfg), int(n_sm), int(batch), None, None, C.byref(n_tasks),
                         C.byref(n_bars)), "mk_plan")
    tasks = np.empty((n_tasks.value, 32), dtype=np.int32)
    off = np.empty(n_sm + 1, dtype=np.int32)
    _check(lib().mk_plan(C.byref(cfg), int(n_sm), int(batch), _ptr(tasks), _ptr(off), None, None),
           "mk_plan")
    return tasks, off, n_bars.value


def mk_plan_step(cfg: mk_config, n_sm: int, batch: int, seq_lens) -> dict:
    """The host schedule of one step (see include/mk.h): task lists, split-KV
    items and the counter-target SM counts."""
    sl = _i32(seq_lens)
    info = np.zeros(9, dtype=np.int32)
    _check(lib().mk_plan_step(C.byref(cfg), int(n_sm), int(batch), _ptr(sl), _ptr(info), None, None,
                              None, None, None), "mk_plan_step")
    n_tasks, n_items = int(info[0]), int(info[1])
    tasks = np.zeros((n_tasks, 32), dtype=np.int32)
    task_off = np.zeros(n_sm + 1, dtype=np.int32)
    items = np.zeros((max(n_items, 1), 8), dtype=np.int32)
    item_off = np.zeros(n_sm + 1, dtype=np.int32)
    meta = np.zeros((batch, 2), dtype=np.int32)
    _check(lib().mk_plan_step(C.byref(cfg), int(n_sm), int(batch), _ptr(sl), _ptr(info), _ptr(tasks),
                              _ptr(task_off), _ptr(items), _ptr(item_off), _ptr(meta)), "mk_plan_step")
    return {"tasks": tasks, "task_off": task_off, "items": items[:n_items], "item_off": item_off,
            "meta": meta, "n_attn": int(info[2]), "n_comb_sms": int(info[3]), "n_up_sms": int(info[4]),
            "n_down_sms": int(info[5]), "n_rtr_sms": int(info[6]), "split": int(info[7]),
            "n_bars": int(info[8])}


def mk_read_trace(h) -> np.ndarray:
    size = C.c_size_t(0)
    _check(lib().mk_read_trace(h, None, 0, C.byref(size)), "mk_read_trace")
    out = np.empty(size.value // 4, dtype=np.int32)
    _check(lib().mk_read_trace(h, _ptr(out), size.value, None), "mk_read_trace")
    return out.reshape(-1, 16)


def mk_read_debug(h, which: int) -> np.ndarray:
    size = C.c_size_t(0)
    _check(lib().mk_read_debug(h, int(which), None, 0, C.byref(size)), "mk_read_debug")
    out = np.empty(size.value // 4, dtype=np.int32)
    _check(lib().mk_read_debug(h, int(which), _ptr(out), size.value, None), "mk_read_debug")
    return out


def mk_debug_bump_wait(h, layer: int, delta: int) -> int:
    return _check(lib().mk_debug_bump_wait(h, int(layer), int(delta)), "mk_debug_bump_wait")


def mk_device_bytes(h) -> int:
    return int(lib().mk_device_bytes(h))


def mk_num_sms(h) -> int:
    return int(lib().mk_num_sms(h))


def mk_step_upload_bytes(h, batch: int) -> int:
    return int(lib().mk_step_upload_bytes(h, int(batch)))


def mk_destroy(h) -> None:
    if h:
        lib().mk_destroy(h)


def mk_service_create(h, logits_ptr: int):
    s = C.c_void_p()
    _check(lib().mk_service_create(h, C.c_void_p(int(logits_ptr)), C.byref(s)), "mk_service_create")
    return s


def mk_service_submit(s, pages, cached_len: int, first_token: int, max_new_tokens: int) -> int:
    pg = _i32(pages)
    rid = C.c_int64(0)
    _check(lib().mk_service_submit(s, _ptr(pg), int(pg.size), int(cached_len), int(first_token),
                                   int(max_new_tokens), C.byref(rid)), "mk_service_submit")
    return int(rid.value)


def mk_service_run(s, n_steps: int) -> int:
    return _check(lib().mk_service_run(s, int(n_steps)), "mk_service_run")


def mk_service_wait(s) -> int:
    return _check(lib().mk_service_wait(s), "mk_service_wait")


def mk_service_result(s, rid: int, cap: int = 4096):
    out = np.empty(cap, dtype=np.int32)
    n, done = C.c_int(0), C.c_int(0)
    _check(lib().mk_service_result(s, C.c_int64(rid), _ptr(out), int(cap), C.byref(n), C.byref(done)),
           "mk_service_result")
    return out[:min(n.value, cap)].copy(), bool(done.value)


def mk_service_batch(s, max_batch: int):
    ids = np.zeros(max_batch, dtype=np.int64)
    lens = np.zeros(max_batch, dtype=np.int32)
    toks = np.zeros(max_batch, dtype=np.int32)
    b = C.c_int(0)
    _check(lib().mk_service_batch(s, _ptr(ids), _ptr(lens), _ptr(toks), C.byref(b)), "mk_service_batch")
    return ids[:b.value].copy(), lens[:b.value].copy(), toks[:b.value].copy()


def mk_service_destroy(s) -> None:
    if s:
        lib().mk_service_destroy(s)


# ---------------------------------------------------------- convenience

def make_config(dims, max_batch: int, max_pages_per_seq: int, num_kv_pages: int, **kw) -> mk_config:
    """mk_config from a ModelDims plus capacity / schedule fields."""
    c = mk_config(n_layers=dims.n_layers, hidden=dims.hidden, n_q_heads=dims.n_q_heads,
                  n_kv_heads=dims.n_kv_heads, head_dim=dims.head_dim, n_experts=dims.n_experts,
                  top_k=dims.top_k, moe_inter=dims.moe_inter, vocab=dims.vocab,
                  page_size=dims.page_size, rope_theta=float(dims.rope_theta),
                  rms_eps=float(dims.rms_eps), max_batch=int(max_batch),
                  max_pages_per_seq=int(max_pages_per_seq), num_kv_pages=int(num_kv_pages))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


class Decoder:
    """Owns one mk handle over caller-owned device tensors (weights, KV pools).

    ``model`` has the stacked BF16 device tensors of ``synth.SynthModel``;
    ``k_pool`` / ``v_pool`` are [L, pages, hkv, P, d] BF16 device tensors.
    The tensors are kept referenced for the lifetime of the decoder.
    """

    def __init__(self, model, k_pool, v_pool, max_batch: int, max_pages_per_seq: int, **cfg_kw):
        self.dims = model.dims
        self.model, self.k_pool, self.v_pool = model, k_pool, v_pool
        L = self.dims.n_layers
        fp8 = getattr(model, "fp8", None)
        if fp8 is not None:
            cfg_kw = {**cfg_kw, "expert_format": MK_EXPERTS_FP8_E4M3}
        self.cfg = make_config(self.dims, max_batch, max_pages_per_seq, k_pool.shape[1], **cfg_kw)
        self._keep = []

        def arr(t):
            a = (C.c_void_p * L)(*[t[l].data_ptr() for l in range(L)])
            self._keep.append(a)
            return C.cast(a, _VPP)

        ex = fp8 if fp8 is not None else {"q_gate": model.w_gate, "q_up": model.w_up, "q_down": model.w_down}
        self.weights = mk_weights(embed=model.embed.data_ptr(), lm_head=model.lm_head.data_ptr(),
                                  final_norm=model.final_norm.data_ptr(),
                                  attn_norm=arr(model.attn_norm), w_qkv=arr(model.w_qkv),
                                  w_o=arr(model.w_o), w_router=arr(model.w_router),
                                  w_gate=arr(ex["q_gate"]), w_up=arr(ex["q_up"]),
                                  w_down=arr(ex["q_down"]), k_pool=arr(k_pool), v_pool=arr(v_pool))
        if fp8 is not None:
            self.weights.s_gate = arr(fp8["s_gate"])
            self.weights.s_up = arr(fp8["s_up"])
            self.weights.s_down = arr(fp8["s_down"])
        self.h = mk_create(self.cfg, self.weights)
        self.batch = 0

    def schedule(self, tokens, page_tables, seq_lens, seq_ids=None, stream=None):
        self.batch = len(tokens)
        pt = _i32(page_tables)
        if pt.shape[1] != self.cfg.max_pages_per_seq:
            full = np.full((pt.shape[0], self.cfg.max_pages_per_seq), -1, dtype=np.int32)
            full[:, :pt.shape[1]] = pt
            pt = full
        return mk_schedule_step(self.h, self.batch, seq_ids, tokens, pt, seq_lens, stream)

    def decode(self, logits, stream=None):
        return mk_decode_step(self.h, logits.data_ptr(), stream)

    def decode_static(self, logits, stream=None):
        return mk_decode_step_static(self.h, logits.data_ptr(), stream)

    def status(self):
        return mk_step_status(self.h)

    def routing(self):
        return mk_get_routing(self.h, self.dims.n_layers, self.batch, self.dims.top_k)

    def trace(self) -> np.ndarray:
        return mk_read_trace(self.h)

    def scratch(self, which: int, layer: int) -> bytes:
        return mk_read_scratch(self.h, which, layer)

    def close(self):
        if self.h:
            mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
