"""ctypes binding over libtfq.so (include/tfq.h), same names as the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
library. Tensors are torch tensors on a CUDA device; bf16 activations may be
``torch.bfloat16`` or 16-bit integer tensors holding bf16 bit patterns. The
library is required: importing this module without a built ``libtfq.so``
raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

TF_OK = 0
TF_E_INVALID_ARG = 1
TF_E_UNSUPPORTED_SHAPE = 2
TF_E_WORKSPACE_TOO_SMALL = 3
TF_E_BAD_PACK = 4
TF_E_CUDA = 5
TF_E_TIMEOUT = 6
TF_E_INTERNAL = 7
TF_DTYPE_BF16 = 0
TF_DTYPE_F32 = 1
TF_RUN_PDL = 1
TF_QWEIGHT_MAGIC = 0x31515446
TF_PACK_VERSION = 2
TF_CODE_AFFINE = 0
TF_CODE_NVFP4 = 1
TF_TUNE_ROWBLOCKS = 0
TF_TUNE_SPLITK = 1
TF_TUNE_STAGE_GROUPS = 2
TF_TUNE_STAGES = 3
TF_TUNE_WARPS = 4
TF_TUNE_MODE = 5
TF_TUNE_CHAIN = 6

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int32
SZ = ctypes.c_size_t


class tf_qweight(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("bits", I32), ("group", I32),
                ("code", I32), ("global_scale", ctypes.c_float), ("batch", I64), ("N", I64), ("K", I64), ("n_pad", I64), ("tile_bytes", I64),
                ("matrix_bytes", I64), ("data", P)]


class tf_decoder_layer(ctypes.Structure):
    _fields_ = [("qkv", tf_qweight), ("o", tf_qweight), ("gate", tf_qweight), ("up", tf_qweight),
                ("down", tf_qweight), ("attn_norm", P), ("mlp_norm", P)]


class tf_decoder_desc(ctypes.Structure):
    _fields_ = [("n_layers", I32), ("d_model", I64), ("d_ff", I64), ("q_dim", I64), ("kv_dim", I64),
                ("vocab", I64), ("eps", ctypes.c_float), ("layers", ctypes.POINTER(tf_decoder_layer)),
                ("final_norm", P), ("readout", tf_qweight)]


class TfqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{status_str(status)}: {msg}")
        self.status = status


_lib = None

# name -> (restype, argtypes); mirrors include/tfq.h
_SIGS = {
    "tf_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "tf_last_error": (ctypes.c_char_p, []),
    "tf_version": (ctypes.c_int, []),
    "tf_qlinear_packed_bytes": (SZ, [I64, I64, I64, ctypes.c_int, ctypes.c_int]),
    "tf_qlinear_pack": (ctypes.c_int, [P, P, P, I64, I64, I64, ctypes.c_int, ctypes.c_int, P, SZ,
                                       ctypes.POINTER(tf_qweight), P]),
    "tf_qlinear_pack_nvfp4": (ctypes.c_int, [P, P, ctypes.c_float, I64, I64, P, SZ, ctypes.POINTER(tf_qweight), P]),
    "tf_qlinear_pack_nvfp4_experts": (ctypes.c_int, [P, P, P, I64, I64, I64, P, SZ, ctypes.POINTER(tf_qweight), P]),
    "tf_qlinear_unpack_debug": (ctypes.c_int, [ctypes.POINTER(tf_qweight), P, P, P, P]),
    "tf_qweight_check": (ctypes.c_int, [ctypes.POINTER(tf_qweight), P]),
    "tf_qlinear_workspace_bytes": (SZ, [ctypes.POINTER(tf_qweight), I64]),
    "tf_qlinear_run": (ctypes.c_int, [ctypes.POINTER(tf_qweight), P, I64, I64, P, ctypes.c_float, P, P,
                                      ctypes.c_int, P, SZ, ctypes.c_uint, P]),
    "tf_qlinear_run_rht": (ctypes.c_int, [ctypes.POINTER(tf_qweight), P, I64, I64, P, P, ctypes.c_float, P, P,
                                          ctypes.c_int, P, ctypes.c_size_t, ctypes.c_uint, P]),
    "tf_qlinear_run_noalloc": (ctypes.c_int, [ctypes.POINTER(tf_qweight), P, I64, I64, P, ctypes.c_float, P, P,
                                              ctypes.c_int, ctypes.c_uint, P]),
    "tf_qlinear_noalloc_status": (ctypes.c_int, [P]),
    "tf_qmlp_gateup_workspace_bytes": (SZ, [ctypes.POINTER(tf_qweight), ctypes.POINTER(tf_qweight), I64]),
    "tf_qmlp_gateup_run": (ctypes.c_int, [ctypes.POINTER(tf_qweight), ctypes.POINTER(tf_qweight), P, I64, I64,
                                          P, ctypes.c_float, P, P, SZ, ctypes.c_uint, P]),
    "tf_qmoe_workspace_bytes": (SZ, [ctypes.POINTER(tf_qweight)] * 3 + [I64, ctypes.c_int]),
    "tf_qmoe_run": (ctypes.c_int, [ctypes.POINTER(tf_qweight)] * 3 + [P, I64, ctypes.c_int, P, P, P, P, P, SZ,
                                                                        ctypes.c_uint, P]),
    "tf_decode_step_workspace_bytes": (SZ, [ctypes.POINTER(tf_decoder_desc), I64]),
    "tf_decode_step_debug_elems": (SZ, [ctypes.POINTER(tf_decoder_desc), I64]),
    "tf_decode_step_run": (ctypes.c_int, [ctypes.POINTER(tf_decoder_desc), P, I64, P, P, SZ, P, ctypes.c_uint,
                                          P]),
    "tf_argmax_rows": (ctypes.c_int, [P, I64, I64, I64, P, P]),
    "tf_embed_rows": (ctypes.c_int, [ctypes.POINTER(tf_qweight), P, I64, P, P, ctypes.c_size_t, P]),
    "tf_draft_prompt_lookup": (I64, [P, I64, P, I64, ctypes.c_int, ctypes.c_int, P]),
    "tf_generate_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tf_decoder_desc)]),
    "tf_generate_greedy": (ctypes.c_int, [ctypes.POINTER(tf_decoder_desc), P, I64, I64, ctypes.c_int, ctypes.c_int, P,
                                          P, P, P, P, ctypes.c_size_t, P]),
    "tf_workspace_status": (ctypes.c_int, [P, P]),
    "tf_selftest_wait_timeout": (ctypes.c_int, [P, ctypes.c_uint64, P]),
    "tf_tune_set": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
}


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libtfq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libtfq.so is not built ({path}); run skinny_gemm_bit_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().tf_status_str(status).decode()


def last_error() -> str:
    return lib().tf_last_error().decode()


def _check(rc: int):
    if rc != TF_OK:
        raise TfqError(rc, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def tune_set(key: int, value: int):
    _check(lib().tf_tune_set(key, value))


# ---------------------------------------------------------------------------- packing

class QWeight:
    """A packed weight buffer (device) and its host descriptor."""

    def __init__(self, buf: torch.Tensor, desc: tf_qweight):
        self.buf = buf
        self.desc = desc

    @property
    def N(self):
        return self.desc.N

    @property
    def K(self):
        return self.desc.K

    @property
    def bits(self):
        return self.desc.bits

    @property
    def batch(self):
        return self.desc.batch

    @property
    def code(self):
        return self.desc.code

    def weight_bytes(self) -> int:
        """Algorithmic bytes of the codes and scales/biases (excluding row padding): 4/64 B a
        weight for a bf16 scale and bias per 64, or 1/16 for an E4M3 scale per 16 (NVFP4)."""
        return int(self.batch * self.N * self.K * (self.bits / 8 + (1 / 16 if self.code == TF_CODE_NVFP4 else 4 / 64)))


def packed_bytes(batch: int, N: int, K: int, bits: int, group: int = 64) -> int:
    return lib().tf_qlinear_packed_bytes(batch, N, K, bits, group)


def _as_dev(a, dtype, device):
    if isinstance(a, torch.Tensor):
        return a.to(device=device).contiguous()
    import numpy as np
    arr = np.ascontiguousarray(a)
    if arr.dtype == np.uint32:
        arr = arr.view(np.int32)
    elif arr.dtype == np.uint16:
        arr = arr.view(np.int16)
    return torch.from_numpy(arr).to(device=device)


def tf_qlinear_pack(wq, scales, biases, bits: int, device="cuda", stream=None) -> QWeight:
    """Pack MLX-layout weights ([B,] N, K*bits/32 uint32; [B,] N, K/64 bf16) into a QWeight."""
    wq = _as_dev(wq, torch.int32, device)
    scales = _as_dev(scales, torch.int16, device)
    biases = _as_dev(biases, torch.int16, device)
    batched = wq.dim() == 3
    batch = wq.shape[0] if batched else 1
    N = wq.shape[-2]
    K = wq.shape[-1] * 32 // bits
    nbytes = packed_bytes(batch, N, K, bits)
    if nbytes == 0:
        raise TfqError(TF_E_UNSUPPORTED_SHAPE, f"unsupported packing N={N} K={K} bits={bits}")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    desc = tf_qweight()
    _check(lib().tf_qlinear_pack(_ptr(wq), _ptr(scales), _ptr(biases), batch, N, K, bits, 64, _ptr(buf), nbytes,
                                 ctypes.byref(desc), _stream(stream)))
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    return QWeight(buf, desc)


def tf_qlinear_pack_nvfp4(codes, block_scales, global_scale, device="cuda", stream=None) -> QWeight:
    """Pack NVFP4 weights (codes uint8 [N, K/2], E4M3 block scales uint8 [N, K/16], fp32
    global scale) into a QWeight; a stack of experts (codes [E, N, K/2], block scales
    [E, N, K/16], global scales fp32 [E]) goes through tf_qlinear_pack_nvfp4_experts."""
    codes = _as_dev(codes, torch.uint8, device)
    block_scales = _as_dev(block_scales, torch.uint8, device)
    experts = codes.dim() == 3
    E = codes.shape[0] if experts else 1
    N, K = codes.shape[-2], codes.shape[-1] * 2
    lead = (E,) if experts else ()
    if codes.dtype != torch.uint8 or block_scales.dtype != torch.uint8 or tuple(block_scales.shape) != lead + (N, K // 16):
        raise TfqError(TF_E_INVALID_ARG, "codes must be uint8 [(E,) N, K/2] and block_scales uint8 [(E,) N, K/16]")
    nbytes = packed_bytes(E, N, K, 4, 16)
    if nbytes == 0:
        raise TfqError(TF_E_UNSUPPORTED_SHAPE, f"unsupported NVFP4 packing N={N} K={K}")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    desc = tf_qweight()
    if experts:
        gs = torch.as_tensor(np.asarray(global_scale, dtype=np.float32).reshape(E)).to(device)
        _check(lib().tf_qlinear_pack_nvfp4_experts(_ptr(codes), _ptr(block_scales), _ptr(gs), E, N, K, _ptr(buf),
                                                   nbytes, ctypes.byref(desc), _stream(stream)))
    else:
        _check(lib().tf_qlinear_pack_nvfp4(_ptr(codes), _ptr(block_scales), float(global_scale), N, K, _ptr(buf),
                                           nbytes, ctypes.byref(desc), _stream(stream)))
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    return QWeight(buf, desc)


def tf_qlinear_unpack_debug(w: QWeight, stream=None):
    """(wq int32, scales int16, biases int16) in MLX layout, read back out of the packed buffer;
    for NVFP4 weights (codes uint8 [(E,) N, K/2], block scales uint8 [(E,) N, K/16], the
    per-matrix fp32 scales [E])."""
    dev = w.buf.device
    if w.code == TF_CODE_NVFP4:
        lead = (w.batch,) if w.batch > 1 else ()
        codes = torch.empty(lead + (w.N, w.K // 2), dtype=torch.uint8, device=dev)
        sc = torch.empty(lead + (w.N, w.K // 16), dtype=torch.uint8, device=dev)
        gs = torch.empty(w.batch, dtype=torch.float32, device=dev)
        _check(lib().tf_qlinear_unpack_debug(ctypes.byref(w.desc), _ptr(codes), _ptr(sc), _ptr(gs), _stream(stream)))
        return codes, sc, gs
    lead = (w.batch,) if w.batch > 1 else ()
    wq = torch.empty(lead + (w.N, w.K * w.bits // 32), dtype=torch.int32, device=dev)
    s = torch.empty(lead + (w.N, w.K // 64), dtype=torch.int16, device=dev)
    b = torch.empty_like(s)
    _check(lib().tf_qlinear_unpack_debug(ctypes.byref(w.desc), _ptr(wq), _ptr(s), _ptr(b), _stream(stream)))
    return wq, s, b


def tf_qweight_check(w: QWeight, stream=None):
    _check(lib().tf_qweight_check(ctypes.byref(w.desc), _stream(stream)))


# ---------------------------------------------------------------------------- workspaces

def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (256-byte aligned by the caching allocator)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def tf_qlinear_workspace_bytes(w: QWeight, M: int = 8) -> int:
    return lib().tf_qlinear_workspace_bytes(ctypes.byref(w.desc), M)


def tf_qmlp_gateup_workspace_bytes(gate: QWeight, up: QWeight, M: int = 8) -> int:
    return lib().tf_qmlp_gateup_workspace_bytes(ctypes.byref(gate.desc), ctypes.byref(up.desc), M)


def tf_qmoe_workspace_bytes(gate: QWeight, up: QWeight, down: QWeight, M: int, top_k: int) -> int:
    return lib().tf_qmoe_workspace_bytes(ctypes.byref(gate.desc), ctypes.byref(up.desc), ctypes.byref(down.desc),
                                         M, top_k)


def tf_workspace_status(ws: torch.Tensor, stream=None) -> int:
    return lib().tf_workspace_status(_ptr(ws), _stream(stream))


def tf_selftest_wait_timeout(ws, limit_ns: int, stream=None):
    """ws=None targets the status word of tf_qlinear_run_noalloc's fixed array."""
    _check(lib().tf_selftest_wait_timeout(_ptr(ws), limit_ns, _stream(stream)))


def tf_qlinear_noalloc_status(stream=None) -> int:
    """Status recorded in tf_qlinear_run_noalloc's fixed array (cleared, with the array, after a failure)."""
    return lib().tf_qlinear_noalloc_status(_stream(stream))


# ---------------------------------------------------------------------------- projections

def _rows(x: torch.Tensor):
    if x.dim() != 2:
        raise ValueError("activations must be 2-D [M, K]")
    return x.shape[0], x.stride(0)


def tf_qlinear_run(w: QWeight, x: torch.Tensor, gamma=None, eps: float = 1e-6, residual=None, out=None,
                   out_dtype=torch.bfloat16, ws=None, flags: int = 0, stream=None) -> torch.Tensor:
    """y = (residual +) rmsnorm?(x) . dequant(W)^T for x [M, K] (M <= 8)."""
    M, ldx = _rows(x)
    if out is None:
        out = torch.empty((M, w.N), dtype=out_dtype, device=x.device)
    ydt = TF_DTYPE_F32 if out.dtype == torch.float32 else TF_DTYPE_BF16
    if ws is None:
        ws = workspace(tf_qlinear_workspace_bytes(w, M), x.device)
    _check(lib().tf_qlinear_run(ctypes.byref(w.desc), _ptr(x), ldx, M, _ptr(gamma), eps, _ptr(residual), _ptr(out),
                                ydt, _ptr(ws), ws.numel(), flags, _stream(stream)))
    return out


def tf_qlinear_run_rht(w: QWeight, x: torch.Tensor, signs: torch.Tensor, gamma=None, eps: float = 1e-6,
                       residual=None, out=None, out_dtype=torch.bfloat16, ws=None, flags: int = 0,
                       stream=None) -> torch.Tensor:
    """tf_qlinear_run with the input Hadamard transform: signs is a device uint8 [K / 8] bit vector."""
    M, ldx = _rows(x)
    if signs.dtype != torch.uint8 or not signs.is_cuda or signs.numel() * 8 < w.K:
        raise ValueError("signs must be a device uint8 tensor of K / 8 bytes")
    if out is None:
        out = torch.empty((M, w.N), dtype=out_dtype, device=x.device)
    ydt = TF_DTYPE_F32 if out.dtype == torch.float32 else TF_DTYPE_BF16
    if ws is None:
        ws = workspace(tf_qlinear_workspace_bytes(w, M), x.device)
    _check(lib().tf_qlinear_run_rht(ctypes.byref(w.desc), _ptr(x), ldx, M, _ptr(signs), _ptr(gamma), eps,
                                    _ptr(residual), _ptr(out), ydt, _ptr(ws), ws.numel(), flags, _stream(stream)))
    return out


def tf_qlinear_run_noalloc(w: QWeight, x: torch.Tensor, gamma=None, eps: float = 1e-6, residual=None, out=None,
                           out_dtype=torch.bfloat16, flags: int = 0, stream=None) -> torch.Tensor:
    """tf_qlinear_run with the library's fixed scratch array instead of a workspace."""
    M, ldx = _rows(x)
    if out is None:
        out = torch.empty((M, w.N), dtype=out_dtype, device=x.device)
    ydt = TF_DTYPE_F32 if out.dtype == torch.float32 else TF_DTYPE_BF16
    _check(lib().tf_qlinear_run_noalloc(ctypes.byref(w.desc), _ptr(x), ldx, M, _ptr(gamma), eps, _ptr(residual),
                                        _ptr(out), ydt, flags, _stream(stream)))
    return out


def tf_qmlp_gateup_run(gate: QWeight, up: QWeight, x: torch.Tensor, gamma=None, eps: float = 1e-6, out=None,
                       ws=None, flags: int = 0, stream=None) -> torch.Tensor:
    """h = silu(xn . G^T) * (xn . U^T), xn = rmsnorm(x) when gamma is given."""
    M, ldx = _rows(x)
    if out is None:
        out = torch.empty((M, gate.N), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(tf_qmlp_gateup_workspace_bytes(gate, up, M), x.device)
    _check(lib().tf_qmlp_gateup_run(ctypes.byref(gate.desc), ctypes.byref(up.desc), _ptr(x), ldx, M, _ptr(gamma),
                                    eps, _ptr(out), _ptr(ws), ws.numel(), flags, _stream(stream)))
    return out


def tf_qmoe_run(gate: QWeight, up: QWeight, down: QWeight, logits: torch.Tensor, x: torch.Tensor, top_k: int,
                out=None, idx=None, wts=None, ws=None, flags: int = 0, stream=None):
    """(y [M, H] bf16, topk_idx [M, k] int32, topk_w [M, k] fp32)."""
    M = x.shape[0]
    dev = x.device
    if out is None:
        out = torch.empty((M, gate.K), dtype=torch.bfloat16, device=dev)
    if idx is None:
        idx = torch.empty((M, top_k), dtype=torch.int32, device=dev)
    if wts is None:
        wts = torch.empty((M, top_k), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(tf_qmoe_workspace_bytes(gate, up, down, M, top_k), dev)
    _check(lib().tf_qmoe_run(ctypes.byref(gate.desc), ctypes.byref(up.desc), ctypes.byref(down.desc), _ptr(logits),
                             M, top_k, _ptr(x), _ptr(out), _ptr(idx), _ptr(wts), _ptr(ws), ws.numel(), flags,
                             _stream(stream)))
    return out, idx, wts


# ---------------------------------------------------------------------------- decoder step

class Decoder:
    """Packed weights of a dense decoder's projections and the host descriptor over them."""

    def __init__(self, layers, final_norm: torch.Tensor, readout: QWeight, d_model: int, d_ff: int, q_dim: int,
                 kv_dim: int, eps: float = 1e-6):
        self.layers = layers            # list of dicts: qkv, o, gate, up, down (QWeight), attn_norm, mlp_norm
        self.final_norm = final_norm
        self.readout = readout
        arr = (tf_decoder_layer * max(1, len(layers)))()
        for i, L in enumerate(layers):
            arr[i].qkv = L["qkv"].desc
            arr[i].o = L["o"].desc
            arr[i].gate = L["gate"].desc
            arr[i].up = L["up"].desc
            arr[i].down = L["down"].desc
            arr[i].attn_norm = L["attn_norm"].data_ptr()
            arr[i].mlp_norm = L["mlp_norm"].data_ptr()
        self._arr = arr
        d = tf_decoder_desc()
        d.n_layers = len(layers)
        d.d_model, d.d_ff, d.q_dim, d.kv_dim, d.vocab = d_model, d_ff, q_dim, kv_dim, readout.N
        d.eps = eps
        d.layers = ctypes.cast(arr, ctypes.POINTER(tf_decoder_layer))
        d.final_norm = final_norm.data_ptr()
        d.readout = readout.desc
        self.desc = d

    def weight_bytes(self) -> int:
        total = self.readout.weight_bytes()
        for L in self.layers:
            total += sum(L[k].weight_bytes() for k in ("qkv", "o", "gate", "up", "down"))
        return total


def tf_decode_step_workspace_bytes(dec: Decoder, M: int) -> int:
    return lib().tf_decode_step_workspace_bytes(ctypes.byref(dec.desc), M)


def tf_decode_step_debug_elems(dec: Decoder, M: int) -> int:
    return lib().tf_decode_step_debug_elems(ctypes.byref(dec.desc), M)


def tf_decode_step_run(dec: Decoder, x: torch.Tensor, out=None, ws=None, debug=None, flags: int = 0,
                       stream=None) -> torch.Tensor:
    """logits [M, vocab] bf16 of one decoder step over the residual stream x [M, d_model]."""
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, dec.readout.N), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(tf_decode_step_workspace_bytes(dec, M), x.device)
    _check(lib().tf_decode_step_run(ctypes.byref(dec.desc), _ptr(x), M, _ptr(out), _ptr(ws), ws.numel(),
                                    _ptr(debug), flags, _stream(stream)))
    return out


# ---------------------------------------------------------------- verify block

def tf_argmax_rows(v: torch.Tensor, stream=None) -> torch.Tensor:
    """idx[m] = lowest index of the largest value of row m of a bf16 [M, N] tensor."""
    M, N = v.shape
    idx = torch.empty(M, dtype=torch.int32, device=v.device)
    _check(lib().tf_argmax_rows(_ptr(v), v.stride(0), M, N, _ptr(idx), _stream(stream)))
    return idx


def tf_embed_rows(w: QWeight, ids: torch.Tensor, ws=None, stream=None) -> torch.Tensor:
    """bf16 [M, K]: the dequantised rows ids (device int32 [M]) of a packed matrix."""
    M = ids.numel()
    out = torch.empty((M, w.K), dtype=torch.bfloat16, device=ids.device)
    if ws is None:
        ws = workspace(256, ids.device)
    _check(lib().tf_embed_rows(ctypes.byref(w.desc), _ptr(ids), M, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def tf_draft_prompt_lookup(prompt, tail, max_ngram: int = 3, max_draft: int = 7):
    """The draft (list of ints) the prompt proposes after the tail (host only)."""
    p = np.ascontiguousarray(prompt, dtype=np.int32)
    t = np.ascontiguousarray(tail, dtype=np.int32)
    d = np.zeros(max(1, max_draft), dtype=np.int32)
    n = lib().tf_draft_prompt_lookup(p.ctypes.data, p.size, t.ctypes.data, t.size, max_ngram, max_draft, d.ctypes.data)
    if n < 0:
        raise TfqError(TF_E_INVALID_ARG, "tf_draft_prompt_lookup: bad arguments")
    return d[:n].tolist()


def tf_generate_workspace_bytes(dec: Decoder) -> int:
    return lib().tf_generate_workspace_bytes(ctypes.byref(dec.desc))


def tf_generate_greedy(dec: Decoder, prompt, max_new: int, max_draft: int = 7, max_ngram: int = 3, ws=None,
                       stream=None):
    """(tokens, steps, drafts kept) of greedy generation with a verify block."""
    p = np.ascontiguousarray(prompt, dtype=np.int32)
    out = np.zeros(max(1, max_new), dtype=np.int32)
    n_out, n_steps, n_acc = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    if ws is None:
        ws = workspace(tf_generate_workspace_bytes(dec))
    _check(lib().tf_generate_greedy(ctypes.byref(dec.desc), p.ctypes.data, p.size, max_new, max_draft, max_ngram,
                                    out.ctypes.data, ctypes.byref(n_out), ctypes.byref(n_steps), ctypes.byref(n_acc),
                                    _ptr(ws), ws.numel(), _stream(stream)))
    return out[:n_out.value].tolist(), n_steps.value, n_acc.value
