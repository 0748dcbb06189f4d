"""Thin ctypes binding of the C ABI (include/tee.h, include/tee_ops.h).

Argument marshalling only: every step of the encoder runs in the CUDA
library.  There is no fallback: if the compiled library is missing, loading
raises.  Device buffers are passed as raw pointers (``tensor.data_ptr()``),
streams as ``torch.cuda.Stream.cuda_stream`` integers.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

TEE_OK = 0
TEE_EINVAL = -1
TEE_ENOTLOADED = -2
TEE_ENOMEM = -3
TEE_ECUDA = -4
TEE_ETOOLONG = -5
TEE_ETIMEOUT = -6

TEE_F32, TEE_BF16, TEE_W8A8, TEE_W4A8, TEE_W6A8 = 0, 1, 2, 3, 4
DTYPES = {"fp32": TEE_F32, "bf16": TEE_BF16, "w8a8": TEE_W8A8, "w4a8": TEE_W4A8, "w6a8": TEE_W6A8}

TEE_LN_ATTN, TEE_LN_MLP = 0, 1
TEE_W_QKV, TEE_W_OUT, TEE_W_FFN_IN, TEE_W_FFN_OUT = 0, 1, 2, 3

KERNEL_CLASSES = ["embed", "layernorm", "gemm", "attention", "elementwise", "pool", "quant"]


class TeeConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("intermediate", ctypes.c_int), ("vocab", ctypes.c_int),
        ("global_every", ctypes.c_int), ("window", ctypes.c_int),
        ("rope_base_global", ctypes.c_float), ("rope_base_local", ctypes.c_float), ("ln_eps", ctypes.c_float),
        ("dtype", ctypes.c_int), ("max_tokens", ctypes.c_int), ("max_texts", ctypes.c_int),
        ("emb_norm", ctypes.c_int), ("final_norm", ctypes.c_int), ("proj_dim", ctypes.c_int),
    ]


_FP = ctypes.POINTER(ctypes.c_float)
_FPP = ctypes.POINTER(_FP)


class TeeWeights(ctypes.Structure):
    _fields_ = [("tok_emb", _FP), ("ln_attn", _FPP), ("wqkv", _FPP), ("wo", _FPP),
                ("ln_mlp", _FPP), ("wi", _FPP), ("wo_ffn", _FPP),
                ("ln_emb", _FP), ("ln_final", _FP), ("w_proj", _FP)]


class TeeKernelStat(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64), ("total_ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


_vp = ctypes.c_void_p
_i = ctypes.c_int
_ctx = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)

# name -> (restype, argtypes), for every function declared in include/*.h
SIGNATURES = {
    "tee_create": (_i, [ctypes.POINTER(TeeConfig), _i, ctypes.POINTER(_ctx)]),
    "tee_load_weights": (_i, [_ctx, ctypes.POINTER(TeeWeights)]),
    "tee_encode": (_i, [_ctx, _vp, _vp, _i, _vp]),
    "tee_encode_device": (_i, [_ctx, _vp, _vp, _vp, _i, _vp, _vp]),
    "tee_encode_tokens": (_i, [_ctx, _vp, _vp, _i, _vp]),
    "tee_encode_tokens_device": (_i, [_ctx, _vp, _vp, _vp, _i, _vp, _vp]),
    "tee_last_error": (ctypes.c_char_p, [_ctx]),
    "tee_destroy": (None, [_ctx]),
    "tee_profile_enable": (_i, [_ctx, _i]),
    "tee_profile_read": (_i, [_ctx, ctypes.POINTER(TeeKernelStat)]),
    "tee_op_embed": (_i, [_ctx, _vp, _i, _vp, _vp]),
    "tee_op_positions": (_i, [_ctx, _vp, _vp, _i, _vp, _vp]),
    "tee_op_layernorm": (_i, [_ctx, _i, _i, _vp, _vp, _i, _vp]),
    "tee_op_qkv": (_i, [_ctx, _i, _vp, _vp, _vp, _i, _vp]),
    "tee_op_attention": (_i, [_ctx, _i, _vp, _vp, _vp, _i, _vp, _vp]),
    "tee_op_out_proj": (_i, [_ctx, _i, _vp, _vp, _i, _vp]),
    "tee_op_ffn_in": (_i, [_ctx, _i, _vp, _vp, _i, _vp]),
    "tee_op_ffn_out": (_i, [_ctx, _i, _vp, _vp, _i, _vp]),
    "tee_op_pool_l2": (_i, [_ctx, _vp, _vp, _vp, _i, _vp, _vp]),
    "tee_op_gemm_bf16": (_i, [_ctx, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "tee_op_quant_rows7": (_i, [_ctx, _vp, _i, _i, _vp, _vp, _vp]),
    "tee_op_w8a8_partials": (_i, [_ctx, _i, _i, _vp, _i, _vp, _vp]),
    "tee_weight_codes": (_i, [_ctx, _i, _i, _vp, _vp]),
    "tee_device_status": (_i, [_ctx]),
    "tee_pool_l2_noalloc": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp]),
    "tee_selftest_wait_timeout": (_i, [_ctx, ctypes.c_longlong, _vp]),
    "tee_selftest_gelu": (_i, [_vp, _vp, ctypes.c_longlong, _vp]),
    "tee_plan_attention": (_i, [_vp, _i, _i, _i, _vp, _i]),
    "tee_plan_attention_schedule": (_i, [_vp, _i, _i, _i, _vp, _vp]),
    "tee_unigram_create": (_i, [ctypes.POINTER(ctypes.c_char_p), _vp, _i, _i, ctypes.c_float, _i, _i,
                                ctypes.POINTER(_vp)]),
    "tee_unigram_encode": (_i, [_vp, ctypes.c_char_p, _i, _vp, _i]),
    "tee_unigram_destroy": (None, [_vp]),
    "tee_similarity": (_i, [_vp, _i, _i, _vp]),
    "tee_plan_gemm": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
}

_LIB = None


class TeeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"tee error {code}: {msg}")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled library (built by ``__graft_entry__.build()``).  Raises if absent."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _ptr(a) -> int:
    """Device or host pointer of a torch tensor / numpy array / int."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if isinstance(a, np.ndarray):
        if not a.flags.c_contiguous:
            raise ValueError("array must be C-contiguous")
        return a.ctypes.data
    raise TypeError(type(a))


def config_from_shape(shape, dtype: str, max_tokens: int, max_texts: int) -> TeeConfig:
    return TeeConfig(shape.n_layers, shape.hidden, shape.n_heads, shape.head_dim, shape.intermediate, shape.vocab,
                     shape.global_every, shape.window, shape.rope_base_global, shape.rope_base_local,
                     shape.ln_eps, DTYPES[dtype], int(max_tokens), int(max_texts),
                     int(getattr(shape, "emb_norm", False)), int(getattr(shape, "final_norm", False)),
                     int(getattr(shape, "proj_dim", 0)))


class Encoder:
    """One library context: owns device weights and workspace."""

    def __init__(self, shape, dtype: str = "bf16", max_tokens: int = 32768, max_texts: int = 4096, device: int = 0):
        self.lib = load()
        self.shape = shape
        self.dtype = dtype
        self.cfg = config_from_shape(shape, dtype, max_tokens, max_texts)
        ctx = ctypes.c_void_p()
        rc = self.lib.tee_create(ctypes.byref(self.cfg), device, ctypes.byref(ctx))
        if rc != TEE_OK:
            raise TeeError(rc, self.lib.tee_last_error(None).decode())
        self.ctx = ctx

    # -- helpers --------------------------------------------------------
    def check(self, rc):
        if rc != TEE_OK:
            raise TeeError(rc, self.lib.tee_last_error(self.ctx).decode())
        return rc

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.tee_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- public API -------------------------------------------------------
    def load_weights(self, w):
        L = self.shape.n_layers
        keep = []

        def f32(a):
            a = np.ascontiguousarray(a, dtype=np.float32)
            keep.append(a)
            return a.ctypes.data_as(_FP)

        def arr(lst):
            ptrs = (_FP * L)(*[f32(a) for a in lst])
            keep.append(ptrs)
            return ctypes.cast(ptrs, _FPP)

        def opt(a):
            return f32(a) if a is not None else None

        tw = TeeWeights(f32(w.tok_emb), arr(w.ln_attn), arr(w.wqkv), arr(w.wo), arr(w.ln_mlp), arr(w.wi),
                        arr(w.wo_ffn), opt(getattr(w, "ln_emb", None)), opt(getattr(w, "ln_final", None)),
                        opt(getattr(w, "w_proj", None)))
        self.check(self.lib.tee_load_weights(self.ctx, ctypes.byref(tw)))

    def encode(self, ids, cu_seqlens) -> np.ndarray:
        """Host arrays in, host fp32 [n, H] out (synchronous)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        n = cu.shape[0] - 1
        out = np.empty((max(n, 0), self.shape.hidden), dtype=np.float32)
        self.check(self.lib.tee_encode(self.ctx, ids.ctypes.data, cu.ctypes.data, n, out.ctypes.data))
        return out

    def encode_device(self, d_ids, d_cu, h_cu, d_out, stream=0):
        h_cu = np.ascontiguousarray(h_cu, dtype=np.int32)
        self.check(self.lib.tee_encode_device(self.ctx, _ptr(d_ids), _ptr(d_cu), h_cu.ctypes.data,
                                              h_cu.shape[0] - 1, _ptr(d_out), stream))

    @property
    def token_width(self) -> int:
        """Width D of the per-token output: proj_dim, else hidden."""
        return int(getattr(self.shape, "proj_dim", 0)) or self.shape.hidden

    def encode_tokens(self, ids, cu_seqlens) -> np.ndarray:
        """Host arrays in, host fp32 [T, D] per-token unit vectors out (synchronous)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        out = np.empty((int(cu[-1]) if cu.shape[0] else 0, self.token_width), dtype=np.float32)
        self.check(self.lib.tee_encode_tokens(self.ctx, ids.ctypes.data, cu.ctypes.data, cu.shape[0] - 1,
                                              out.ctypes.data))
        return out

    def encode_tokens_device(self, d_ids, d_cu, h_cu, d_out, stream=0):
        h_cu = np.ascontiguousarray(h_cu, dtype=np.int32)
        self.check(self.lib.tee_encode_tokens_device(self.ctx, _ptr(d_ids), _ptr(d_cu), h_cu.ctypes.data,
                                                     h_cu.shape[0] - 1, _ptr(d_out), stream))

    def profile_enable(self, on=True):
        self.check(self.lib.tee_profile_enable(self.ctx, 1 if on else 0))

    def profile_read(self) -> dict:
        stats = (TeeKernelStat * len(KERNEL_CLASSES))()
        self.check(self.lib.tee_profile_read(self.ctx, stats))
        return {name: {"launches": s.launches, "total_ms": s.total_ms, "flops": s.flops, "bytes": s.bytes}
                for name, s in zip(KERNEL_CLASSES, stats)}

    def device_status(self) -> int:
        return self.lib.tee_device_status(self.ctx)

    # -- per-step entry points (tee_ops.h) ------------------------------
    def op(self, name, *args):
        return self.check(getattr(self.lib, name)(self.ctx, *[_ptr(a) if not isinstance(a, (int, float)) else a
                                                              for a in args]))


# ---------------------------------------------------------------------------
# host-side front end (tee_frontend.h)
# ---------------------------------------------------------------------------

class Unigram:
    """Unigram max-score segmenter over a vocabulary (tee_unigram_*).

    ``pieces``: list of str (piece i has id i); ``scores``: their scores;
    ``unk_id`` / ``unk_score``: the unknown piece for uncovered characters;
    ``bos_id`` / ``eos_id``: ids wrapped around every text (-1 for none).
    """

    def __init__(self, pieces, scores, unk_id: int, unk_score: float, bos_id: int = -1, eos_id: int = -1):
        self.lib = load()
        enc = [p.encode("utf-8") for p in pieces]
        arr = (ctypes.c_char_p * len(enc))(*enc)
        sc = np.ascontiguousarray(scores, dtype=np.float32)
        if sc.shape != (len(enc),):
            raise ValueError("one score per piece")
        h = ctypes.c_void_p()
        rc = self.lib.tee_unigram_create(arr, sc.ctypes.data, len(enc), unk_id, unk_score, bos_id, eos_id,
                                         ctypes.byref(h))
        if rc != TEE_OK:
            raise TeeError(rc, self.lib.tee_last_error(None).decode())
        self.h = h

    def encode(self, text: str) -> np.ndarray:
        raw = text.encode("utf-8")
        n = self.lib.tee_unigram_encode(self.h, raw, len(raw), None, 0)
        if n < 0:
            raise TeeError(n, self.lib.tee_last_error(None).decode())
        ids = np.empty(n, dtype=np.int32)
        n2 = self.lib.tee_unigram_encode(self.h, raw, len(raw), ids.ctypes.data, n)
        if n2 != n:
            raise TeeError(n2, self.lib.tee_last_error(None).decode())
        return ids

    def close(self):
        if getattr(self, "h", None):
            self.lib.tee_unigram_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pack_texts(id_lists):
    """Pack per-text id arrays into one batch: (ids int32[T], cu_seqlens int32[n + 1])."""
    lens = [len(a) for a in id_lists]
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    ids = np.concatenate([np.asarray(a, np.int32) for a in id_lists]) if id_lists else np.zeros(0, np.int32)
    return ids, cu


def similarity(vecs) -> np.ndarray:
    """The [n, n] matrix of dot products of the rows of ``vecs`` (tee_similarity)."""
    lib = load()
    v = np.ascontiguousarray(vecs, dtype=np.float32)
    n, dim = v.shape
    out = np.empty((n, n), dtype=np.float32)
    rc = lib.tee_similarity(v.ctypes.data, n, dim, out.ctypes.data)
    if rc != TEE_OK:
        raise TeeError(rc, lib.tee_last_error(None).decode())
    return out


def format_similarity(sim) -> str:
    """The matrix as the `-sim` listing prints it: one row per line, four decimals."""
    return "\n".join(" ".join(f"{x:.4f}" for x in row) for row in np.asarray(sim))
