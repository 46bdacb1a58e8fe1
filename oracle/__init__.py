"""CPU oracle of the persistent MoE decode step (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It imports
nothing from the CUDA product package: both sides meet only through the
seeded synthetic inputs.

The arithmetic lives in ``oracle.c`` (fp64 on BF16 inputs); this module only
marshals numpy arrays.  Every function cites its passage in the C source.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liboracle.so")
# a prebuilt copy of the same source to load instead (the sanitizer test
# builds one with AddressSanitizer); it is used as it is, never rebuilt
LIB_OVERRIDE = os.environ.get("ORACLE_LIB")

BF16_X, BF16_Q, BF16_ATTN, BF16_A = 1, 2, 4, 8
ALL_BF16 = BF16_X | BF16_Q | BF16_ATTN | BF16_A

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, portable flags)."""
    src = os.path.join(HERE, "oracle.c")
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(HERE, "oracle.h"))):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wno-maybe-uninitialized",
                    "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class _Dims(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads",
                                         "head_dim", "n_experts", "top_k", "moe_inter",
                                         "vocab", "page_size", "num_pages")] + \
               [("rope_theta", C.c_double), ("rms_eps", C.c_double)]


_PP = C.POINTER(C.c_void_p)


class _Fp8(C.Structure):
    _fields_ = [(n, _PP) for n in ("q_gate", "q_up", "q_down", "s_gate", "s_up", "s_down")]


class _Model(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("attn_norm", _PP), ("w_qkv", _PP), ("w_o", _PP), ("w_router", _PP),
                ("w_gate", _PP), ("w_up", _PP), ("w_down", _PP),
                ("k_pool", _PP), ("v_pool", _PP), ("fp8", C.POINTER(_Fp8))]


class _Trace(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("h_in", "x", "q", "attn", "attn_proj", "router",
                                           "idx", "w", "gap", "moe", "xf")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if LIB_OVERRIDE:
                L = C.CDLL(LIB_OVERRIDE)
            else:
                build()
                L = C.CDLL(LIB_PATH)
            vp, i32, dbl = C.c_void_p, C.c_int, C.c_double
            L.orc_bf16_to_double.restype = dbl
            L.orc_bf16_to_double.argtypes = [C.c_uint16]
            L.orc_double_to_bf16.restype = C.c_uint16
            L.orc_double_to_bf16.argtypes = [dbl]
            L.orc_round_bf16.restype = dbl
            L.orc_round_bf16.argtypes = [dbl]
            L.orc_rmsnorm.argtypes = [i32, vp, vp, dbl, vp]
            L.orc_rope.argtypes = [i32, vp, C.c_long, dbl]
            L.orc_matvec.argtypes = [i32, i32, vp, i32, vp, vp]
            L.orc_e4m3_to_double.restype = dbl
            L.orc_e4m3_to_double.argtypes = [C.c_uint8]
            L.orc_matvec_e4m3.argtypes = [i32, i32, vp, vp, vp, vp]
            L.orc_paged_attention.argtypes = [C.POINTER(_Dims), vp, vp, vp, i32, i32, vp, vp]
            L.orc_paged_attention.restype = i32
            L.orc_route.argtypes = [i32, i32, vp, vp, vp, vp]
            L.orc_moe.argtypes = [C.POINTER(_Dims), C.POINTER(_Model), i32, vp, i32, vp, vp,
                                  C.c_uint, vp]
            L.orc_decode_step.argtypes = [C.POINTER(_Dims), C.POINTER(_Model), i32, vp, vp, vp,
                                          i32, C.c_uint, vp, C.POINTER(_Trace)]
            L.orc_decode_step.restype = i32
            L.orc_decode_step_forced.argtypes = [C.POINTER(_Dims), C.POINTER(_Model), i32, vp, vp, vp,
                                                 i32, C.c_uint, vp, vp, vp, C.POINTER(_Trace)]
            L.orc_decode_step_forced.restype = i32
            L.orc_run_layers.argtypes = [C.POINTER(_Dims), C.POINTER(_Model), i32, i32, i32,
                                         vp, vp, i32, C.c_uint, vp]
            L.orc_run_layers.restype = i32
            L.orc_set_threads.argtypes = [i32]
            L.orc_get_threads.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == np.uint16, "BF16 inputs are passed as uint16 bit patterns"
    assert a.flags.c_contiguous
    return a


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# ---------------------------------------------------------------- pieces

def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x: float) -> float:
    return float(lib().orc_round_bf16(float(x)))


def to_bf16_bits(x) -> np.ndarray:
    x = _f64(x)
    out = np.empty(x.shape, dtype=np.uint16)
    f = lib().orc_double_to_bf16
    for i, v in enumerate(x.reshape(-1)):
        out.reshape(-1)[i] = f(float(v))
    return out


def rmsnorm(h, gain_bits, eps: float) -> np.ndarray:
    h = _f64(h)
    g = _u16(np.ascontiguousarray(gain_bits))
    out = np.empty_like(h)
    lib().orc_rmsnorm(h.size, _p(h), _p(g), float(eps), _p(out))
    return out


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = _f64(v).copy()
    lib().orc_rope(v.size, _p(v), int(pos), float(theta))
    return v


def matvec(w_bits, x) -> np.ndarray:
    w = _u16(np.ascontiguousarray(w_bits))
    x = _f64(x)
    rows, cols = w.shape
    nvec = 1 if x.ndim == 1 else x.shape[0]
    y = np.empty((nvec, rows), dtype=np.float64)
    lib().orc_matvec(rows, cols, _p(w), nvec, _p(x), _p(y))
    return y[0] if x.ndim == 1 else y


def e4m3_to_f64(codes) -> np.ndarray:
    """OCP E4M3 byte -> value (orc_e4m3_to_double), elementwise."""
    c = np.asarray(codes, dtype=np.uint8)
    f = lib().orc_e4m3_to_double
    return np.array([f(int(v)) for v in c.reshape(-1)], dtype=np.float64).reshape(c.shape)


def matvec_e4m3(q, scale, x) -> np.ndarray:
    """y[r] = sum_c (scale[r] * e4m3(q[r][c])) * x[c] (orc_matvec_e4m3)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sc = np.ascontiguousarray(scale, dtype=np.float32)
    x = _f64(x)
    rows, cols = q.shape
    assert sc.shape == (rows,) and x.shape == (cols,)
    y = np.empty(rows, dtype=np.float64)
    lib().orc_matvec_e4m3(rows, cols, _p(q), _p(sc), _p(x), _p(y))
    return y


def _dims(d: dict, num_pages: int) -> _Dims:
    return _Dims(n_layers=d["n_layers"], hidden=d["hidden"], n_q_heads=d["n_q_heads"],
                 n_kv_heads=d["n_kv_heads"], head_dim=d["head_dim"], n_experts=d["n_experts"],
                 top_k=d["top_k"], moe_inter=d["moe_inter"], vocab=d["vocab"],
                 page_size=d["page_size"], num_pages=num_pages,
                 rope_theta=float(d["rope_theta"]), rms_eps=float(d["rms_eps"]))


def paged_attention(dims: dict, k_pool_l, v_pool_l, page_table, n_keys: int, kv_head: int,
                    q) -> np.ndarray:
    """One query head over one layer's paged pools ([pages, hkv, P, d] uint16)."""
    k = _u16(k_pool_l)
    v = _u16(v_pool_l)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    q = _f64(q)
    out = np.empty(dims["head_dim"], dtype=np.float64)
    dm = _dims(dims, k.shape[0])
    rc = lib().orc_paged_attention(C.byref(dm), _p(k), _p(v), _p(pt), int(n_keys), int(kv_head),
                                   _p(q), _p(out))
    if rc != 0:
        raise RuntimeError(f"orc_paged_attention failed: {rc}")
    return out


def route(logits, top_k: int):
    r = _f64(logits)
    idx = np.empty(top_k, dtype=np.int32)
    w = np.empty(top_k, dtype=np.float64)
    gap = np.empty(1, dtype=np.float64)
    lib().orc_route(r.size, top_k, _p(r), _p(idx), _p(w), _p(gap))
    return idx, w, float(gap[0])


# ------------------------------------------------------------ the model

class Oracle:
    """Host model: BF16 weights (uint16 views, stacked over layers) + its own KV pools.

    ``weights`` maps the names embed, lm_head, final_norm, attn_norm, w_qkv, w_o,
    w_router, w_gate, w_up, w_down to uint16 arrays with the layouts given in
    oracle.h (stacked over a leading layer axis where per-layer).  ``k_pool`` /
    ``v_pool`` are [L, pages, hkv, P, d] uint16 arrays that the oracle appends
    the new K/V to (the caller keeps ownership).

    ``fp8``, if given, maps q_gate, q_up, q_down (uint8 E4M3 codes, [L, E, I,
    H] / [L, E, H, I]) and s_gate, s_up, s_down (float32 per-row scales, [L,
    E, I] / [L, E, H]) to arrays: the routed experts then use those weights
    (orc_fp8_experts) and w_gate / w_up / w_down may be omitted.
    """

    PER_LAYER = ("attn_norm", "w_qkv", "w_o", "w_router", "w_gate", "w_up", "w_down")
    FP8 = ("q_gate", "q_up", "q_down", "s_gate", "s_up", "s_down")

    def __init__(self, dims: dict, weights: dict, k_pool: np.ndarray, v_pool: np.ndarray,
                 fp8: dict | None = None):
        self.dims = dict(dims)
        weights = dict(weights)
        if fp8 is not None:
            for n in ("w_gate", "w_up", "w_down"):
                weights.setdefault(n, np.zeros((self.dims["n_layers"], 1), dtype=np.uint16))
        self.w = {n: _u16(a) for n, a in weights.items()}
        self.k_pool = _u16(k_pool)
        self.v_pool = _u16(v_pool)
        L = self.dims["n_layers"]
        self.num_pages = int(self.k_pool.shape[1])
        self._dm = _dims(self.dims, self.num_pages)
        self._arrays = []

        def ptrs(arr):
            assert arr.shape[0] >= L
            base = arr.ctypes.data
            stride = arr.strides[0]
            a = (C.c_void_p * L)(*[base + i * stride for i in range(L)])
            self._arrays.append(a)
            return C.cast(a, _PP)

        self._m = _Model(embed=self.w["embed"].ctypes.data, lm_head=self.w["lm_head"].ctypes.data,
                         final_norm=self.w["final_norm"].ctypes.data,
                         **{n: ptrs(self.w[n]) for n in self.PER_LAYER},
                         k_pool=ptrs(self.k_pool), v_pool=ptrs(self.v_pool))
        self.fp8 = None
        if fp8 is not None:
            E, I, H = self.dims["n_experts"], self.dims["moe_inter"], self.dims["hidden"]
            shapes = {"q_gate": (E, I, H), "q_up": (E, I, H), "q_down": (E, H, I),
                      "s_gate": (E, I), "s_up": (E, I), "s_down": (E, H)}
            self.fp8 = {}
            for n in self.FP8:
                a = np.asarray(fp8[n])
                assert a.dtype == (np.uint8 if n[0] == "q" else np.float32) and a.flags.c_contiguous, n
                assert a.shape[1:] == shapes[n] and a.shape[0] >= L, n
                self.fp8[n] = a
            self._f8 = _Fp8(**{n: ptrs(self.fp8[n]) for n in self.FP8})
            self._m.fp8 = C.pointer(self._f8)

    def moe(self, layer: int, x, idx, w, flags: int = 0) -> np.ndarray:
        x = _f64(x)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        w = _f64(w)
        assert idx.shape == w.shape and idx.ndim == 1
        assert np.all((idx >= 0) & (idx < self.dims["n_experts"]))
        out = np.empty(self.dims["hidden"], dtype=np.float64)
        lib().orc_moe(C.byref(self._dm), C.byref(self._m), int(layer), _p(x), int(idx.size), _p(idx),
                      _p(w), int(flags), _p(out))
        return out

    def decode_step(self, tokens, seq_lens, page_tables, flags: int = 0, trace: bool = False,
                    force=None):
        """One step; ``force`` = (idx int32 [L, B, k], mask bool [L, B]) imposes
        those experts where mask is set (orc_decode_step_forced)."""
        d = self.dims
        B = len(tokens)
        L, H, E, K = d["n_layers"], d["hidden"], d["n_experts"], d["top_k"]
        QD = d["n_q_heads"] * d["head_dim"]
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        pt = np.ascontiguousarray(page_tables, dtype=np.int32)
        assert pt.ndim == 2 and pt.shape[0] == B
        logits = np.empty((B, d["vocab"]), dtype=np.float64)
        tr = None
        out = {}
        if trace:
            out = {"h_in": np.zeros((L + 1, B, H)), "x": np.zeros((L, B, H)),
                   "q": np.zeros((L, B, QD)), "attn": np.zeros((L, B, QD)),
                   "attn_proj": np.zeros((L, B, H)), "router": np.zeros((L, B, E)),
                   "idx": np.zeros((L, B, K), dtype=np.int32), "w": np.zeros((L, B, K)),
                   "gap": np.zeros((L, B)), "moe": np.zeros((L, B, H)),
                   "xf": np.zeros((B, H))}
            tr = _Trace(**{n: a.ctypes.data for n, a in out.items()})
        if force is not None:
            fidx = np.ascontiguousarray(force[0], dtype=np.int32)
            fmask = np.ascontiguousarray(force[1], dtype=np.uint8)
            assert fidx.shape == (L, B, K) and fmask.shape == (L, B)
            rc = lib().orc_decode_step_forced(C.byref(self._dm), C.byref(self._m), B, _p(tok), _p(sl),
                                              _p(pt), pt.shape[1], int(flags), _p(fidx), _p(fmask),
                                              _p(logits), C.byref(tr) if tr is not None else None)
        else:
            rc = lib().orc_decode_step(C.byref(self._dm), C.byref(self._m), B, _p(tok), _p(sl),
                                       _p(pt), pt.shape[1], int(flags), _p(logits),
                                       C.byref(tr) if tr is not None else None)
        if rc != 0:
            raise RuntimeError(f"orc_decode_step failed: {rc}")
        return (logits, out) if trace else logits

    def run_layers(self, l0: int, l1: int, h, seq_lens, page_tables, flags: int = 0) -> np.ndarray:
        h = _f64(h).copy()
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        pt = np.ascontiguousarray(page_tables, dtype=np.int32)
        rc = lib().orc_run_layers(C.byref(self._dm), C.byref(self._m), int(l0), int(l1),
                                  h.shape[0], _p(sl), _p(pt), pt.shape[1], int(flags), _p(h))
        if rc != 0:
            raise RuntimeError(f"orc_run_layers failed: {rc}")
        return h
