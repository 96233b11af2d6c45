"""Python binding of libfa.so: the C-ABI entry points under the same names.

Argument marshalling only -- every step of the attention runs in the CUDA
kernels behind the C ABI. Tensors are torch CUDA tensors (torch provides the
device memory and the stream); nothing here computes attention, and there is
no fallback: if the library is missing or the call fails, an exception says so.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "fa.h")

FA_OK = 0
FA_FP16, FA_BF16, FA_FP8_E4M3 = 0, 1, 2
_DTYPE = {torch.float16: FA_FP16, torch.bfloat16: FA_BF16}

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})")


def header_functions():
    """Names of the functions include/fa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", text, flags=re.M)))


def lib():
    """Load libfa.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.fa_fwd.restype = i
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, i, i, i, vp]
        L.fa_fp8_prep.restype = i
        L.fa_fp8_prep.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
        L.fa_fwd_fp8.restype = i
        L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_varlen_blocks.restype = i
        L.fa_varlen_blocks.argtypes = [vp, i, vp, vp]
        L.fa_fp8_prep_varlen.restype = i
        L.fa_fp8_prep_varlen.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, i, i, vp, vp, vp, vp,
                                         i, i, i, i, i, vp]
        L.fa_fwd_fp8_varlen.restype = i
        L.fa_fwd_fp8_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, vp, vp, vp, vp, i, i, i, i, i,
                                        f, i, vp]
        L.fa_fwd_paged.restype = i
        L.fa_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, i, i, vp,
                                   ctypes.c_size_t, i, vp]
        L.fa_bwd_workspace_size.restype = ctypes.c_size_t
        L.fa_bwd_workspace_size.argtypes = [i, i]
        L.fa_bwd.restype = i
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, i, i, vp,
                             ctypes.c_size_t, i, vp]
        L.fa_fwd_splitkv_workspace_size.restype = ctypes.c_size_t
        L.fa_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i, i]
        L.fa_fwd_splitkv.restype = i
        L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, ctypes.c_size_t, i, vp]
        L.fa_get_device_status.restype = i
        L.fa_get_device_status.argtypes = [vp, ctypes.POINTER(i)]
        L.fa_strerror.restype = ctypes.c_char_p
        L.fa_strerror.argtypes = [i]
        L.fa_version.restype = i
        L.fa_version.argtypes = []
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().fa_strerror(int(status)).decode()


def fa_version() -> int:
    return lib().fa_version()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def fa_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, cu_seqlens_q=None, cu_seqlens_k=None,
           total_q=0, total_k=0, dtype=None, stream=None, check=True) -> int:
    """Raw entry point: pointers from the tensors, sizes as given. Returns the
    status; raises FAError when ``check`` and the status is not FA_OK."""
    if dtype is None:
        dtype = _DTYPE[q.dtype]
    st = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(Sq), int(Sk),
                      int(D), float(scale), int(bool(causal)), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                      int(total_q), int(total_k), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fwd")
    return st


def fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, num_splits) -> int:
    return int(lib().fa_fwd_splitkv_workspace_size(int(B), int(H), int(Sq), int(Sk), int(D), int(num_splits)))


def fa_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, num_splits, workspace, workspace_bytes,
                   dtype=None, stream=None, check=True) -> int:
    """Raw entry point: split-KV forward with a caller-owned workspace."""
    if dtype is None:
        dtype = _DTYPE[q.dtype]
    st = lib().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(Sq), int(Sk),
                              int(D), float(scale), int(bool(causal)), int(num_splits), _ptr(workspace),
                              int(workspace_bytes), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fwd_splitkv")
    return st


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, num_splits, dtype=None,
                           stream=None, check=True) -> int:
    """Raw entry point: split-KV forward whose scratch is the library's own
    fixed array, for callers that cannot allocate device memory."""
    L = lib()
    fn = L.fa_fwd_splitkv_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.restype = i
    fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, i, vp]
    if dtype is None:
        dtype = _DTYPE[q.dtype]
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(Sq), int(Sk), int(D), float(scale),
            int(bool(causal)), int(num_splits), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fwd_splitkv_noalloc")
    return st


def attention_forward_splitkv(q, k, v, *, batch, causal=False, scale=None, num_splits=0, workspace=None,
                              out=None, lse=None, stream=None):
    """Allocate O, LSE and (unless given) the workspace with torch and call
    ``fa_fwd_splitkv``. q ``[B*Sq, H, D]``, k/v ``[B*Sk, H, D]``."""
    B = batch
    H, D = q.shape[1], q.shape[2]
    Sq, Sk = q.shape[0] // B, k.shape[0] // B
    if scale is None:
        scale = D ** -0.5
    nbytes = fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, num_splits)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), device=q.device, dtype=torch.float32)
    fa_fwd_splitkv(q, k, v, out, lse, B, H, Sq, Sk, D, scale, causal, num_splits, workspace,
                   workspace.numel() * workspace.element_size(), stream=stream)
    return out, lse


def fa_fp8_prep(q, k, v, q8, k8, v8, q_scale, k_scale, v_scale, sigma, B, H, Sq, Sk, D, in_dtype=None,
                stream=None, check=True) -> int:
    """Raw entry point: Hadamard rotation (``sigma`` int8 +-1, or None for
    none) and per-128-row-block e4m3 quantisation of Q, K (rotated) and V."""
    if in_dtype is None:
        in_dtype = _DTYPE[q.dtype]
    st = lib().fa_fp8_prep(_ptr(q), _ptr(k), _ptr(v), int(in_dtype), _ptr(q8), _ptr(k8), _ptr(v8),
                           _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr(sigma), int(B), int(H), int(Sq),
                           int(Sk), int(D), _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fp8_prep")
    return st


def fa_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, Sq, Sk, D, scale, causal, stream=None,
               check=True) -> int:
    """Raw entry point: attention on e4m3 codes with block scales; bf16 O."""
    st = lib().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr(o),
                          _ptr(lse), int(B), int(H), int(Sq), int(Sk), int(D), float(scale), int(bool(causal)),
                          _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return st


def fa_varlen_blocks(cu_seqlens, B, cu_blocks, stream=None, check=True) -> int:
    """Raw entry point: cu_blocks[b] = sum of ceil(L / 128) over the first b sequences."""
    st = lib().fa_varlen_blocks(_ptr(cu_seqlens), int(B), _ptr(cu_blocks), _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_varlen_blocks")
    return st


def fa_fp8_prep_varlen(q, k, v, q8, k8, v8, q_scale, k_scale, v_scale, sigma, B, H, cu_seqlens_q,
                       cu_seqlens_k, cu_blocks_q, cu_blocks_k, total_q, total_k, max_seqlen_q, max_seqlen_k, D,
                       in_dtype=None, stream=None, check=True) -> int:
    """Raw entry point: ``fa_fp8_prep`` over packed variable-length sequences."""
    if in_dtype is None:
        in_dtype = _DTYPE[(q if q is not None else k).dtype]
    st = lib().fa_fp8_prep_varlen(_ptr(q), _ptr(k), _ptr(v), int(in_dtype), _ptr(q8), _ptr(k8), _ptr(v8),
                                  _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr(sigma), int(B), int(H),
                                  _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(cu_blocks_q), _ptr(cu_blocks_k),
                                  int(total_q), int(total_k), int(max_seqlen_q), int(max_seqlen_k), int(D),
                                  _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fp8_prep_varlen")
    return st


def fa_fwd_fp8_varlen(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, cu_seqlens_q, cu_seqlens_k,
                      cu_blocks_q, cu_blocks_k, total_q, total_k, max_seqlen_q, max_seqlen_k, D, scale, causal,
                      stream=None, check=True) -> int:
    """Raw entry point: ``fa_fwd_fp8`` over packed variable-length sequences."""
    st = lib().fa_fwd_fp8_varlen(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                 _ptr(o), _ptr(lse), int(B), int(H), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                 _ptr(cu_blocks_q), _ptr(cu_blocks_k), int(total_q), int(total_k),
                                 int(max_seqlen_q), int(max_seqlen_k), int(D), float(scale), int(bool(causal)),
                                 _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fwd_fp8_varlen")
    return st


def _fp8_side_varlen(x, cu, H, dev, stream, names):
    """e4m3 codes, block offsets and scale arrays of one packed side."""
    B = cu.numel() - 1
    total = x.shape[0]
    cb = torch.empty(B + 1, dtype=torch.int32, device=dev)
    fa_varlen_blocks(cu, B, cb, stream=stream)
    nb = total // 128 + B   # upper bound on cu_blocks[B]
    out = {n: torch.empty((nb, H), dtype=torch.float32, device=dev) for n in names[1:]}
    out[names[0]] = cb
    return out


def fp8_prepare_varlen(q, k, v, sigma, *, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, stream=None):
    """Varlen ``fp8_prepare``: q ``[total_q, H, D]``, k/v ``[total_k, H, D]``
    16-bit, ``cu_seqlens_*`` int32 CUDA tensors. Either side may be None (q,
    or k and v): that side is skipped, so a K/V cache is prepared once and
    reused. Scale arrays ``[n_blocks, H]`` are allocated at their upper bound
    ``total // 128 + B`` rows; the first ``cu_blocks[B]`` rows are written."""
    ref = q if q is not None else k
    H, D = ref.shape[1], ref.shape[2]
    dev = ref.device
    B = (cu_seqlens_q if cu_seqlens_q is not None else cu_seqlens_k).numel() - 1
    out = {"B": B, "H": H, "D": D, "varlen": True}
    if q is not None:
        out.update(_fp8_side_varlen(q, cu_seqlens_q, H, dev, stream, ("cu_blocks_q", "q_scale")))
        out.update(q8=torch.empty(q.shape, dtype=torch.uint8, device=dev), cu_seqlens_q=cu_seqlens_q,
                   total_q=q.shape[0], max_seqlen_q=max_seqlen_q)
    if k is not None:
        out.update(_fp8_side_varlen(k, cu_seqlens_k, H, dev, stream, ("cu_blocks_k", "k_scale", "v_scale")))
        out.update(k8=torch.empty(k.shape, dtype=torch.uint8, device=dev),
                   v8=torch.empty(v.shape, dtype=torch.uint8, device=dev), cu_seqlens_k=cu_seqlens_k,
                   total_k=k.shape[0], max_seqlen_k=max_seqlen_k)
    g = out.get
    fa_fp8_prep_varlen(q, k, v, g("q8"), g("k8"), g("v8"), g("q_scale"), g("k_scale"), g("v_scale"), sigma, B, H,
                       g("cu_seqlens_q"), g("cu_seqlens_k"), g("cu_blocks_q"), g("cu_blocks_k"), g("total_q", 0),
                       g("total_k", 0), g("max_seqlen_q", 0) if q is not None else 0,
                       g("max_seqlen_k", 0) if k is not None else 0, D,
                       in_dtype=_DTYPE[ref.dtype], stream=stream)
    return out


def fp8_prepare(q, k, v, sigma, *, batch, stream=None):
    """Allocate the e4m3 tensors and block scales and call ``fa_fp8_prep``.
    q ``[B*Sq, H, D]``, k/v ``[B*Sk, H, D]`` 16-bit. Returns a dict."""
    B = batch
    H, D = q.shape[1], q.shape[2]
    Sq, Sk = q.shape[0] // B, k.shape[0] // B
    dev = q.device
    out = {"q8": torch.empty(q.shape, dtype=torch.uint8, device=dev),
           "k8": torch.empty(k.shape, dtype=torch.uint8, device=dev),
           "v8": torch.empty(v.shape, dtype=torch.uint8, device=dev),
           "q_scale": torch.empty((B, H, (Sq + 127) // 128), dtype=torch.float32, device=dev),
           "k_scale": torch.empty((B, H, (Sk + 127) // 128), dtype=torch.float32, device=dev),
           "v_scale": torch.empty((B, H, (Sk + 127) // 128), dtype=torch.float32, device=dev),
           "B": B, "H": H, "Sq": Sq, "Sk": Sk, "D": D}
    fa_fp8_prep(q, k, v, out["q8"], out["k8"], out["v8"], out["q_scale"], out["k_scale"], out["v_scale"],
                sigma, B, H, Sq, Sk, D, stream=stream)
    return out


def fp8_attention_forward(prep, *, causal=False, scale=None, out=None, lse=None, stream=None):
    """Attention on the output of ``fp8_prepare`` (or of ``fp8_prepare_varlen``,
    or a dict merging a Q preparation with a K/V one); returns (O bf16, LSE
    fp32 ``[B, H, Sq]``, varlen ``[H, total_q]``)."""
    if prep.get("varlen"):
        p = prep
        H, D = p["H"], p["D"]
        if scale is None:
            scale = D ** -0.5
        dev = p["q8"].device
        if out is None:
            out = torch.empty((p["total_q"], H, D), dtype=torch.bfloat16, device=dev)
        if lse is None:
            lse = torch.empty((H, p["total_q"]), dtype=torch.float32, device=dev)
        fa_fwd_fp8_varlen(p["q8"], p["k8"], p["v8"], p["q_scale"], p["k_scale"], p["v_scale"], out, lse, p["B"], H,
                          p["cu_seqlens_q"], p["cu_seqlens_k"], p["cu_blocks_q"], p["cu_blocks_k"], p["total_q"],
                          p["total_k"], p["max_seqlen_q"], p["max_seqlen_k"], D, scale, causal, stream=stream)
        return out, lse
    B, H, Sq, Sk, D = prep["B"], prep["H"], prep["Sq"], prep["Sk"], prep["D"]
    if scale is None:
        scale = D ** -0.5
    dev = prep["q8"].device
    if out is None:
        out = torch.empty((B * Sq, H, D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    fa_fwd_fp8(prep["q8"], prep["k8"], prep["v8"], prep["q_scale"], prep["k_scale"], prep["v_scale"], out, lse,
               B, H, Sq, Sk, D, scale, causal, stream=stream)
    return out, lse


def fa_get_device_status(stream=None, check=True):
    raw = ctypes.c_int(0)
    st = lib().fa_get_device_status(_stream(stream), ctypes.byref(raw))
    if check and st != FA_OK:
        raise FAError(st, f"device status word 0x{raw.value:x}")
    return st, raw.value


def attention_forward(q, k, v, *, causal=False, scale=None, cu_seqlens_q=None, cu_seqlens_k=None,
                      max_seqlen_q=None, max_seqlen_k=None, batch=None, out=None, lse=None, stream=None):
    """Allocate O and LSE and call ``fa_fwd``.

    Fixed length: q ``[B*Sq, H, D]`` (or ``[B, Sq, H, D]``), k/v likewise; give
    ``batch`` when passing the flattened form. Varlen: ``cu_seqlens_*`` int32
    CUDA tensors and ``max_seqlen_*``. Returns (O, LSE) with LSE fp32
    ``[B, H, Sq]`` (fixed) or ``[H, total_q]`` (varlen).
    """
    if q.dim() == 4:
        B, Sq, H, D = q.shape
        Sk = k.shape[1]
        q, k, v = q.reshape(B * Sq, H, D), k.reshape(B * Sk, H, D), v.reshape(B * Sk, H, D)
    else:
        H, D = q.shape[1], q.shape[2]
        if cu_seqlens_q is None:
            B = batch
            Sq, Sk = q.shape[0] // B, k.shape[0] // B
        else:
            B = cu_seqlens_q.numel() - 1
            Sq, Sk = max_seqlen_q, max_seqlen_k
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        shape = (H, q.shape[0]) if cu_seqlens_q is not None else (B, H, Sq)
        lse = torch.empty(shape, device=q.device, dtype=torch.float32)
    fa_fwd(q, k, v, out, lse, B, H, Sq, Sk, D, scale, causal, cu_seqlens_q, cu_seqlens_k,
           q.shape[0], k.shape[0], stream=stream)
    return out, lse


def fa_bwd_workspace_size(H, total_q) -> int:
    return int(lib().fa_bwd_workspace_size(int(H), int(total_q)))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Sq, Sk, D, scale, causal, cu_seqlens_q=None,
           cu_seqlens_k=None, total_q=0, total_k=0, workspace=None, workspace_bytes=0, dtype=None, stream=None,
           check=True) -> int:
    """Raw entry point: dQ, dK, dV of the attention forward for upstream gradient dO."""
    if dtype is None:
        dtype = _DTYPE[q.dtype]
    st = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                      int(B), int(H), int(Sq), int(Sk), int(D), float(scale), int(bool(causal)),
                      _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(total_q), int(total_k), _ptr(workspace),
                      int(workspace_bytes), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_bwd")
    return st


def attention_backward(q, k, v, o, lse, dout, *, causal=False, scale=None, cu_seqlens_q=None, cu_seqlens_k=None,
                       max_seqlen_q=None, max_seqlen_k=None, batch=None, workspace=None, stream=None):
    """Allocate dQ, dK, dV (and the scratch) and call ``fa_bwd``. Arguments
    as ``attention_forward``; ``o`` and ``lse`` are its outputs, ``dout`` the
    gradient of ``o``. Returns (dQ, dK, dV)."""
    H, D = q.shape[1], q.shape[2]
    if cu_seqlens_q is None:
        B = batch
        Sq, Sk = q.shape[0] // B, k.shape[0] // B
    else:
        B = cu_seqlens_q.numel() - 1
        Sq, Sk = max_seqlen_q, max_seqlen_k
    if scale is None:
        scale = D ** -0.5
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa_bwd_workspace_size(H, q.shape[0])
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Sq, Sk, D, scale, causal, cu_seqlens_q, cu_seqlens_k,
           q.shape[0], k.shape[0], workspace, workspace.numel() * workspace.element_size(), stream=stream)
    return dq, dk, dv


def fa_fwd_paged(q, k_cache, v_cache, block_table, seqlens_k, o, lse, B, H, Sq, D, num_pages, page_size, max_pages,
                 scale, causal, num_splits=1, workspace=None, workspace_bytes=0, cu_seqlens_q=None, total_q=0,
                 dtype=None, stream=None, check=True) -> int:
    """Raw entry point: attention over K/V held in a paged cache."""
    if dtype is None:
        dtype = _DTYPE[q.dtype]
    st = lib().fa_fwd_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seqlens_k), _ptr(o),
                            _ptr(lse), int(B), int(H), int(Sq), int(D), int(num_pages), int(page_size),
                            int(max_pages), float(scale), int(bool(causal)), _ptr(cu_seqlens_q), int(total_q),
                            int(num_splits), _ptr(workspace), int(workspace_bytes), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FAError(st, "fa_fwd_paged")
    return st


def attention_forward_paged(q, k_cache, v_cache, block_table, seqlens_k, *, causal=False, scale=None, num_splits=1,
                            cu_seqlens_q=None, max_seqlen_q=None, out=None, lse=None, stream=None):
    """Allocate O, LSE (and the split workspace) and call ``fa_fwd_paged``.
    q ``[B*Sq, H, D]`` (or packed ``[total_q, H, D]`` with ``cu_seqlens_q``
    and ``max_seqlen_q``); caches ``[num_pages, page_size, H, D]``;
    block_table int32 ``[B, max_pages]``; seqlens_k int32 ``[B]``. Returns
    (O, LSE ``[B, H, Sq]``, packed ``[H, total_q]``)."""
    B, max_pages = block_table.shape
    num_pages, page_size, H, D = k_cache.shape
    Sq = q.shape[0] // B if cu_seqlens_q is None else max_seqlen_q
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        shape = (B, H, Sq) if cu_seqlens_q is None else (H, q.shape[0])
        lse = torch.empty(shape, device=q.device, dtype=torch.float32)
    ws, ws_bytes = None, 0
    if num_splits != 1:
        ws_bytes = fa_fwd_splitkv_workspace_size(B, H, Sq, max_pages * page_size, D, num_splits)
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    fa_fwd_paged(q, k_cache, v_cache, block_table, seqlens_k, out, lse, B, H, Sq, D, num_pages, page_size, max_pages,
                 scale, causal, num_splits, ws, ws_bytes, cu_seqlens_q=cu_seqlens_q, total_q=q.shape[0],
                 stream=stream)
    return out, lse
