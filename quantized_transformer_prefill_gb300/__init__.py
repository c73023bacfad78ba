"""Python binding of ``libminfer.so`` (the C ABI in ``include/minfer.h``).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  The library must have been built (``build.build()``); there is
no fallback of any kind when it is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB_PATH
_lock = threading.Lock()
_lib = None

MINFER_F32 = 0
MINFER_Q8_0 = 8

ERR_NAMES = {0: "OK", -1: "ERR_ARG", -2: "ERR_POS_OOB", -3: "ERR_TOKEN_OOB",
             -4: "ERR_MISSING_TENSOR", -5: "ERR_SHAPE", -6: "ERR_CUDA", -7: "ERR_OOM",
             -8: "ERR_DEVICE", -9: "ERR_STATE", -10: "ERR_TOO_LARGE"}
# device status codes (minfer_device_status): the bounded wait that gave up
DEV_NAMES = {0: "DEV_OK", 1: "DEV_TIMEOUT_TMA_EMPTY", 2: "DEV_TIMEOUT_MMA_FULL",
             3: "DEV_TIMEOUT_MMA_SLOT", 4: "DEV_TIMEOUT_EPILOGUE", 5: "DEV_TIMEOUT_DRAIN",
             6: "DEV_TIMEOUT_ATTN"}

# every entry point declared in include/minfer.h: name -> (argtypes, restype)
_P, _I, _I64, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float


class Hparams(ctypes.Structure):
    _fields_ = [("n_layer", ctypes.c_int), ("n_embd", ctypes.c_int), ("n_head", ctypes.c_int),
                ("n_head_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("n_ff", ctypes.c_int),
                ("n_vocab", ctypes.c_int), ("max_seq_len", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("tied_embeddings", ctypes.c_int), ("qk_norm", ctypes.c_int)]


class Tensor(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("type", ctypes.c_int), ("ne0", ctypes.c_int64),
                ("ne1", ctypes.c_int64), ("data", ctypes.c_void_p)]


SIGNATURES = {
    "minfer_model_create": ([ctypes.POINTER(Hparams), ctypes.POINTER(_P)], _I),
    "minfer_model_set_tensor": ([_P, ctypes.POINTER(Tensor)], _I),
    "minfer_model_finalize": ([_P], _I),
    "minfer_load_weights": ([ctypes.POINTER(Hparams), ctypes.POINTER(Tensor), _I,
                             ctypes.POINTER(_P)], _I),
    "minfer_free": ([_P], None),
    "minfer_kv_create": ([_P, _I, ctypes.POINTER(_P)], _I),
    "minfer_kv_n_ctx": ([_P], _I),
    "minfer_kv_free": ([_P], None),
    "minfer_kv_read": ([_P, _I, _I, _I, _I, _P], _I),
    "minfer_kv_write": ([_P, _I, _I, _I, _I, _P], _I),
    "minfer_prefill": ([_P, _P, _P, _I, _P, _P], _I),
    "minfer_prefill_device": ([_P, _P, _P, _I, _P, _P, _P], _I),
    "minfer_prefill_n": ([_P, _P, _P, _I, _P, _I, _P], _I),
    "minfer_prefill_device_n": ([_P, _P, _P, _I, _P, _I, _P, _P], _I),
    "minfer_sync_status": ([_P, _P], _I),
    "minfer_set_dump": ([_P, _P, _I], _I),
    "minfer_debug_read": ([_P, ctypes.c_char_p, _P, _I64], _I),
    "minfer_debug_layer": ([_P, _I], _I),
    "minfer_profile_enable": ([_P, _I], _I),
    "minfer_profile_read": ([_P, _I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_I64),
                             ctypes.POINTER(ctypes.c_double)], _I),
    "minfer_op_quantize": ([_P, _I64, _I64, _P, _P], _I),
    "minfer_op_rmsnorm_quantize": ([_P, _P, _I64, _I64, _F, _P, _P], _I),
    "minfer_op_gemm": ([_P, _P, _I64, _P, _P, _I64, _I64, _P, _P], _I),
    "minfer_op_gemm_noalloc": ([_P, _P, _I64, _P, _P, _I64, _I64, _P], _I),
    "minfer_op_gemm_swiglu": ([_P, _P, _I64, _P, _P, _P, _P, _I64, _I64, _P, _P], _I),
    "minfer_op_attention": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P], _I),
    "minfer_op_rope_store": ([_P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P], _I),
    "minfer_op_qknorm_rope_store": ([_P, _P, _P, _P, _F, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P], _I),
    "minfer_strerror": ([_I], ctypes.c_char_p),
    "minfer_device_status": ([_P], _I),
    "minfer_debug_fault": ([_P, _I, _I64], _I),
}


class MinferError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = lib().minfer_strerror(code).decode()
        super().__init__(f"{what}: {ERR_NAMES.get(code, code)} ({msg})")


def lib():
    """The loaded library.  Raises when it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "quantized_transformer_prefill_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def check(rc: int, what: str = "minfer"):
    if rc != 0:
        raise MinferError(rc, what)


def hparams_of(cfg) -> Hparams:
    return Hparams(cfg.n_layer, cfg.n_embd, cfg.n_head, cfg.n_head_kv, cfg.head_dim, cfg.n_ff,
                   cfg.n_vocab, cfg.max_seq_len, cfg.rope_theta, cfg.rms_eps, int(cfg.tied),
                   int(getattr(cfg, "qk_norm", False)))


class Model:
    """A model on the current CUDA device."""

    def __init__(self, hp: Hparams):
        self._hp = hp
        ptr = ctypes.c_void_p()
        check(lib().minfer_model_create(ctypes.byref(hp), ctypes.byref(ptr)), "model_create")
        self.ptr = ptr.value
        self.n_vocab = hp.n_vocab
        self.n_embd = hp.n_embd
        self.n_layer = hp.n_layer
        self._dump = None

    def set_tensor(self, name: str, data: np.ndarray, ne0: int, ne1: int, ttype: int = MINFER_F32):
        data = np.ascontiguousarray(data)
        t = Tensor(name.encode(), ttype, ne0, ne1, data.ctypes.data)
        check(lib().minfer_model_set_tensor(self.ptr, ctypes.byref(t)), f"set_tensor {name}")

    def finalize(self):
        check(lib().minfer_model_finalize(self.ptr), "finalize")

    def kv(self, n_ctx: int) -> "KV":
        return KV(self, n_ctx)

    def prefill(self, kv: "KV", ids: np.ndarray, pos: np.ndarray, out: np.ndarray | None = None):
        """Host-buffer prefill: returns the last token's logits (float32 [V])."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        if out is None:
            out = np.empty(self.n_vocab, np.float32)
        rc = lib().minfer_prefill(self.ptr, ids.ctypes.data, pos.ctypes.data, ids.size, kv.ptr,
                                  out.ctypes.data)
        check(rc, "prefill")
        return out

    def prefill_n(self, kv: "KV", ids: np.ndarray, pos: np.ndarray, n_out: int,
                  out: np.ndarray | None = None):
        """Host-buffer prefill returning the logits of the last n_out tokens
        (float32 [n_out][V], token order)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        if out is None:
            out = np.empty((n_out, self.n_vocab), np.float32)
        check(lib().minfer_prefill_n(self.ptr, ids.ctypes.data, pos.ctypes.data, ids.size, kv.ptr,
                                     n_out, out.ctypes.data), "prefill_n")
        return out

    def prefill_device_n(self, kv: "KV", d_ids: int, d_pos: int, nt: int, n_out: int,
                         d_logits: int, stream: int | None = None) -> int:
        return lib().minfer_prefill_device_n(self.ptr, d_ids, d_pos, nt, kv.ptr, n_out, d_logits,
                                             stream)

    def prefill_rc(self, kv: "KV", ids, pos, out=None) -> int:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        if out is None:
            out = np.empty(self.n_vocab, np.float32)
        return lib().minfer_prefill(self.ptr, ids.ctypes.data, pos.ctypes.data, ids.size, kv.ptr,
                                    out.ctypes.data)

    def prefill_device(self, kv: "KV", d_ids: int, d_pos: int, nt: int, d_logits: int,
                       stream: int | None = None) -> int:
        """Device-buffer prefill enqueued on `stream` (raw cudaStream_t); no sync."""
        return lib().minfer_prefill_device(self.ptr, d_ids, d_pos, nt, kv.ptr, d_logits, stream)

    def sync_status(self, stream: int | None = None) -> int:
        return lib().minfer_sync_status(self.ptr, stream)

    def set_dump(self, buf: np.ndarray | None):
        """buf: float32 [n_layer + 1][max_tokens][n_embd] host array, or None."""
        if buf is None:
            check(lib().minfer_set_dump(self.ptr, None, 0), "set_dump")
            self._dump = None
            return
        assert buf.dtype == np.float32 and buf.flags.c_contiguous
        self._dump = buf
        check(lib().minfer_set_dump(self.ptr, buf.ctypes.data, buf.shape[1]), "set_dump")

    def debug_read(self, name: str, out: np.ndarray) -> np.ndarray:
        check(lib().minfer_debug_read(self.ptr, name.encode(), out.ctypes.data, out.nbytes),
              f"debug_read {name}")
        return out

    def debug_layer(self, layer: int):
        """Capture layer `layer`'s intermediates on the next prefill (-1: off)."""
        check(lib().minfer_debug_layer(self.ptr, layer), "debug_layer")

    def debug_fault(self, layer: int, wait_limit_ns: int = 0):
        """Test hook: layer >= 0 makes that layer's gate/up GEMM withhold one
        operand stage and every GEMM wait give up after wait_limit_ns;
        -1 turns it off."""
        check(lib().minfer_debug_fault(self.ptr, layer, wait_limit_ns), "debug_fault")

    def device_status(self) -> int:
        return lib().minfer_device_status(self.ptr)

    def profile_enable(self, on: bool = True):
        check(lib().minfer_profile_enable(self.ptr, int(on)), "profile_enable")

    def profile_read(self) -> dict:
        out = {}
        k = 0
        while True:
            name = ctypes.c_char_p()
            n = ctypes.c_int64()
            ms = ctypes.c_double()
            if lib().minfer_profile_read(self.ptr, k, ctypes.byref(name), ctypes.byref(n),
                                         ctypes.byref(ms)) != 0:
                break
            out[name.value.decode()] = (int(n.value), float(ms.value))
            k += 1
        return out

    def free(self):
        if getattr(self, "ptr", None):
            lib().minfer_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class KV:
    def __init__(self, model: Model, n_ctx: int):
        ptr = ctypes.c_void_p()
        check(lib().minfer_kv_create(model.ptr, n_ctx, ctypes.byref(ptr)), "kv_create")
        self.ptr = ptr.value
        self.model = model
        self.n_ctx = lib().minfer_kv_n_ctx(self.ptr)
        self.width = model._hp.n_head_kv * model._hp.head_dim

    def read(self, layer: int, which: int, row0: int = 0, nrows: int | None = None) -> np.ndarray:
        nrows = self.n_ctx - row0 if nrows is None else nrows
        out = np.empty((nrows, self.width), np.float32)
        check(lib().minfer_kv_read(self.ptr, layer, which, row0, nrows, out.ctypes.data), "kv_read")
        return out

    def write(self, layer: int, which: int, row0: int, data: np.ndarray):
        data = np.ascontiguousarray(data, dtype=np.float32)
        check(lib().minfer_kv_write(self.ptr, layer, which, row0, data.shape[0], data.ctypes.data),
              "kv_write")

    def free(self):
        if getattr(self, "ptr", None):
            lib().minfer_kv_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def load_model(cfg, tensors) -> Model:
    """Create a model from an iterable of (name, array, ne0, ne1, type)."""
    m = Model(hparams_of(cfg))
    for name, arr, ne0, ne1, ttype in tensors:
        m.set_tensor(name, arr, ne0, ne1, ttype)
    m.finalize()
    return m


# ------------------------------------------------------------------ single stages
# torch tensors (CUDA) in, torch tensors out; the library does the work.

def _ptr(t):
    return t.data_ptr() if t is not None else None


def op_quantize(x):
    import torch
    rows, n = x.shape
    nb = (n + 31) // 32
    q = torch.zeros((rows, nb * 32), dtype=torch.int8, device=x.device)
    d = torch.zeros((rows, nb), dtype=torch.int16, device=x.device)
    check(lib().minfer_op_quantize(_ptr(x.contiguous()), rows, n, _ptr(q), _ptr(d)), "op_quantize")
    return q, d


def op_rmsnorm_quantize(x, w, eps: float):
    import torch
    rows, n = x.shape
    nb = (n + 31) // 32
    q = torch.zeros((rows, nb * 32), dtype=torch.int8, device=x.device)
    d = torch.zeros((rows, nb), dtype=torch.int16, device=x.device)
    check(lib().minfer_op_rmsnorm_quantize(_ptr(x.contiguous()), _ptr(w.contiguous()), rows, n,
                                           eps, _ptr(q), _ptr(d)), "op_rmsnorm_quantize")
    return q, d


def op_gemm(xq, xd, wq, wd, K: int, dots: bool = False):
    import torch
    M, N = xq.shape[0], wq.shape[0]
    nb = (K + 31) // 32
    y = torch.zeros((M, N), dtype=torch.float32, device=xq.device)
    dd = torch.zeros((M, N, nb), dtype=torch.int32, device=xq.device) if dots else None
    check(lib().minfer_op_gemm(_ptr(xq), _ptr(xd), M, _ptr(wq), _ptr(wd), N, K, _ptr(y), _ptr(dd)),
          "op_gemm")
    return (y, dd) if dots else y


def op_gemm_noalloc(xq, xd, wq, wd, K: int):
    """minfer_op_gemm without device allocation (fixed 32 MiB scratch in the
    library).  The call runs on the library's own stream, so the operands
    must be complete when it starts: the current stream is synchronized
    first."""
    import torch
    M, N = xq.shape[0], wq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=xq.device)
    torch.cuda.current_stream(xq.device).synchronize()
    check(lib().minfer_op_gemm_noalloc(_ptr(xq), _ptr(xd), M, _ptr(wq), _ptr(wd), N, K, _ptr(y)),
          "op_gemm_noalloc")
    return y


def op_gemm_swiglu(xq, xd, gq, gd, uq, ud, F: int, K: int):
    import torch
    M = xq.shape[0]
    nbF = (F + 31) // 32
    sq = torch.zeros((M, nbF * 32), dtype=torch.int8, device=xq.device)
    sd = torch.zeros((M, nbF), dtype=torch.int16, device=xq.device)
    check(lib().minfer_op_gemm_swiglu(_ptr(xq), _ptr(xd), M, _ptr(gq), _ptr(gd), _ptr(uq), _ptr(ud),
                                      F, K, _ptr(sq), _ptr(sd)), "op_gemm_swiglu")
    return sq, sd


def op_attention(q, pos, K, V, nh: int, nkv: int, hd: int):
    import torch
    o = torch.zeros_like(q)
    check(lib().minfer_op_attention(_ptr(q), _ptr(pos), q.shape[0], _ptr(K), _ptr(V), K.shape[0],
                                    nh, nkv, hd, _ptr(o)), "op_attention")
    return o


def op_qknorm_rope_store(qkv, bias, qnorm, knorm, eps: float, pos, nh: int, nkv: int, hd: int,
                         theta: float, K, V):
    """RoPE/store with the Qwen3 per-head Q/K RMSNorm first (bias may be None)."""
    import torch
    nt = qkv.shape[0]
    q_out = torch.zeros((nt, nh * hd), dtype=torch.float32, device=qkv.device)
    check(lib().minfer_op_qknorm_rope_store(_ptr(qkv), _ptr(bias), _ptr(qnorm), _ptr(knorm), eps,
                                            _ptr(pos), nt, nh, nkv, hd, theta, K.shape[0],
                                            _ptr(q_out), _ptr(K), _ptr(V)), "op_qknorm_rope_store")
    return q_out


def op_rope_store(qkv, bias, pos, nh: int, nkv: int, hd: int, theta: float, K, V):
    import torch
    nt = qkv.shape[0]
    q_out = torch.zeros((nt, nh * hd), dtype=torch.float32, device=qkv.device)
    check(lib().minfer_op_rope_store(_ptr(qkv), _ptr(bias), _ptr(pos), nt, nh, nkv, hd, theta,
                                     K.shape[0], _ptr(q_out), _ptr(K), _ptr(V)), "op_rope_store")
    return q_out
