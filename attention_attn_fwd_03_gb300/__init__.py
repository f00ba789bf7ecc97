"""GB300-native (sm_103a) exact attention: Python binding of the C ABI in include/attn.h.

Argument marshalling only.  Every step of attention runs in the CUDA library
``libattn_gb300.so`` built in-tree from ``csrc/``; there is no CPU or
PyTorch fallback, and every call raises if the library is missing.

Two levels:
  * ``attn_fwd``, ``attn_fwd_fp8``, ``attn_paged_decode``,
    ``attn_paged_decode_workspace_size``, ``attn_paged_decode_noalloc``,
    ``attn_paged_fwd``, ``attn_paged_fwd_workspace_size``,
    ``attn_varlen_fwd``, ``attn_varlen_fwd_workspace_size``, ``attn_bwd``,
    ``attn_bwd_workspace_size``, ``attn_fwd_host``, ``attn_fwd_host_workspace_size``,
    ``attn_selftest_wait_timeout``, ``attn_selftest_mma_rate``, ``attn_device_status``,
    ``attn_status_string``: the C entry
    points, same names and argument order, taking raw device pointers (ints) and a stream
    handle (int).
  * ``fwd``, ``fwd_fp8``, ``paged_decode``, ``paged_fwd``, ``varlen_fwd``, ``bwd``: take torch CUDA
    tensors, allocate outputs with torch when none are given, call the C entry
    point on the current stream and raise ``AttnError`` on a non-zero status.
  * ``fwd_host``: the same for host (CPU) tensors through ``attn_fwd_host``.
"""
import ctypes
import math
import os
import threading

from . import inputs  # noqa: F401  (seeded synthetic input recipes)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_gb300.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_WORKSPACE = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_DEVICE_DATA = 6

# size of the library's fixed device scratch array used by attn_paged_decode_noalloc
ATTN_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what or "attn", attn_status_string(status), status))


def build(force=False):
    """Compile the CUDA library in-tree (nvcc, sm_103a) and load it."""
    from . import _build
    _build.build(force=force)
    global _lib
    with _lock:
        _lib = None
    return lib()


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("CUDA library %s is missing: build it with "
                                   "attention_attn_fwd_03_gb300.build() (nvcc, sm_103a)" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.attn_fwd.restype = i
            L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
            L.attn_fwd_fp8.restype = i
            L.attn_fwd_fp8.argtypes = [vp, vp, vp, f, f, f, vp, vp, i, i, i, i, i, f, i, vp]
            L.attn_paged_decode_workspace_size.restype = sz
            L.attn_paged_decode_workspace_size.argtypes = [i, i, i, i, i]
            L.attn_paged_decode.restype = i
            L.attn_paged_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp, sz, vp]
            L.attn_paged_decode_noalloc.restype = i
            L.attn_paged_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp]
            L.attn_paged_fwd_workspace_size.restype = sz
            L.attn_paged_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
            L.attn_paged_fwd.restype = i
            L.attn_paged_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, vp, vp, vp, sz,
                                         vp]
            L.attn_varlen_fwd_workspace_size.restype = sz
            L.attn_varlen_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.attn_varlen_fwd.restype = i
            L.attn_varlen_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, vp, vp, sz, vp]
            L.attn_bwd_workspace_size.restype = sz
            L.attn_bwd_workspace_size.argtypes = [i, i, i, i]
            L.attn_bwd.restype = i
            L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
            L.attn_fwd_host_workspace_size.restype = sz
            L.attn_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.attn_fwd_host.restype = i
            L.attn_fwd_host.argtypes = [vp, vp, vp, i, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
            L.attn_selftest_wait_timeout.restype = i
            L.attn_selftest_wait_timeout.argtypes = [vp]
            L.attn_selftest_mma_rate.restype = i
            L.attn_selftest_mma_rate.argtypes = [vp, i, i, vp]
            L.attn_device_status.restype = i
            L.attn_device_status.argtypes = [vp]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_status_string.argtypes = [i]
            _lib = L
        return _lib


# ---------------------------------------------------------------- C entry points

def attn_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream):
    return lib().attn_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream)


def attn_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale, o, lse, B, H, Nq, Nk, d, scale, causal, stream):
    return lib().attn_fwd_fp8(q8, k8, v8, q_descale, k_descale, v_descale, o, lse, B, H, Nq, Nk, d, scale,
                              causal, stream)


def attn_paged_decode_workspace_size(B, H, d, max_pages_per_seq, page_size):
    return lib().attn_paged_decode_workspace_size(B, H, d, max_pages_per_seq, page_size)


def attn_paged_decode(q, k_cache, v_cache, block_table, seq_lens, B, H, d, page_size, max_pages_per_seq,
                      num_pages, scale, o, lse, workspace, workspace_bytes, stream):
    return lib().attn_paged_decode(q, k_cache, v_cache, block_table, seq_lens, B, H, d, page_size,
                                   max_pages_per_seq, num_pages, scale, o, lse, workspace, workspace_bytes,
                                   stream)


def attn_paged_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, B, H, d, page_size,
                              max_pages_per_seq, num_pages, scale, o, lse, stream):
    """Paged decode whose split partials live in the library's fixed device
    scratch array; allocates nothing (see include/attn.h for its limits)."""
    return lib().attn_paged_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, B, H, d, page_size,
                                           max_pages_per_seq, num_pages, scale, o, lse, stream)


def attn_paged_fwd_workspace_size(B, total_q, max_q_len, H, H_kv, d, page_size, max_pages_per_seq):
    return lib().attn_paged_fwd_workspace_size(B, total_q, max_q_len, H, H_kv, d, page_size, max_pages_per_seq)


def attn_paged_fwd(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, B, total_q, max_q_len, H, H_kv, d,
                   page_size, max_pages_per_seq, num_pages, scale, causal, o, lse, workspace, workspace_bytes,
                   stream):
    return lib().attn_paged_fwd(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, B, total_q, max_q_len,
                                H, H_kv, d, page_size, max_pages_per_seq, num_pages, scale, causal, o, lse,
                                workspace, workspace_bytes, stream)


def attn_varlen_fwd_workspace_size(B, total_q, max_q_len, max_k_len, H, H_kv, d):
    return lib().attn_varlen_fwd_workspace_size(B, total_q, max_q_len, max_k_len, H, H_kv, d)


def attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, B, total_q, total_k, max_q_len, max_k_len, H, H_kv, d,
                    scale, causal, o, lse, workspace, workspace_bytes, stream):
    return lib().attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, B, total_q, total_k, max_q_len, max_k_len, H,
                                 H_kv, d, scale, causal, o, lse, workspace, workspace_bytes, stream)


def attn_bwd_workspace_size(B, H, Nq, d):
    return lib().attn_bwd_workspace_size(B, H, Nq, d)


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace, workspace_bytes,
             stream):
    return lib().attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace,
                          workspace_bytes, stream)


def attn_fwd_host_workspace_size(B, H, Nq, Nk, d, n_modes, chunk_bh):
    return lib().attn_fwd_host_workspace_size(B, H, Nq, Nk, d, n_modes, chunk_bh)


def attn_fwd_host(q, k, v, n_modes, causal, o, lse, B, H, Nq, Nk, d, scale, chunk_bh, workspace, workspace_bytes,
                  stream):
    """causal, o and lse are addresses of C arrays of n_modes entries (int, pointer, pointer)."""
    return lib().attn_fwd_host(q, k, v, n_modes, causal, o, lse, B, H, Nq, Nk, d, scale, chunk_bh, workspace,
                               workspace_bytes, stream)


def attn_selftest_wait_timeout(stream):
    return lib().attn_selftest_wait_timeout(stream)


def attn_selftest_mma_rate(cycles, n_ctas, n_groups, stream):
    return lib().attn_selftest_mma_rate(cycles, n_ctas, n_groups, stream)


def attn_device_status(stream):
    return lib().attn_device_status(stream)


def attn_status_string(status):
    return lib().attn_status_string(int(status)).decode()


# ---------------------------------------------------------------- torch helpers

def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(t, name, dtype, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _check_host(t, name, dtype, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError("%s must be a CPU (host) tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _raise(st, what):
    if st != ATTN_OK:
        raise AttnError(st, what)


def fwd(q, k, v, causal=False, scale=None, out=None, lse=None, return_lse=True, stream=None):
    """bf16 [B,H,Nq,d] / [B,H,Nk,d] -> (o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq])."""
    torch = _torch()
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (B, H, Nk, d))
    _check(v, "v", torch.bfloat16, (B, H, Nk, d))
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, q.shape)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, H, Nq))
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    st = attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                  lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, sc, int(bool(causal)),
                  _stream(stream))
    _raise(st, "attn_fwd")
    return out, lse


def fwd_host(q, k, v, causal=(False,), scale=None, out=None, lse=None, chunk_bh=0, workspace=None, stream=None,
             synchronize=True):
    """Host-resident bf16 q [B,H,Nq,d], k, v [B,H,Nk,d] -> (list of o, list of lse), one entry per mask mode
    in ``causal``.  Outputs are page-locked host tensors unless given.  The copies and kernels run on the
    library's chunk pipeline.  With ``synchronize`` (the default) the call returns after synchronising the
    stream, so the outputs are ready; otherwise they are ready once the stream reaches this point."""
    torch = _torch()
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check_host(q, "q", torch.bfloat16)
    _check_host(k, "k", torch.bfloat16, (B, H, Nk, d))
    _check_host(v, "v", torch.bfloat16, (B, H, Nk, d))
    modes = [int(bool(c)) for c in causal]
    n = len(modes)
    if out is None:
        out = [torch.empty(q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    if lse is None:
        lse = [torch.empty((B, H, Nq), dtype=torch.float32).pin_memory() for _ in range(n)]
    if len(out) != n or len(lse) != n:
        raise ValueError("need one out and one lse per mode")
    for m in range(n):
        _check_host(out[m], "out[%d]" % m, torch.bfloat16, q.shape)
        if lse[m] is not None:
            _check_host(lse[m], "lse[%d]" % m, torch.float32, (B, H, Nq))
    need = attn_fwd_host_workspace_size(B, H, Nq, Nk, d, n, chunk_bh)
    if need == 0:
        raise AttnError(ATTN_ERR_INVALID_ARG, "attn_fwd_host_workspace_size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    if workspace.device.type != "cuda" or workspace.numel() < need:
        raise ValueError("workspace must be a CUDA tensor of at least %d bytes" % need)
    c_modes = (ctypes.c_int * n)(*modes)
    c_out = (ctypes.c_void_p * n)(*[t.data_ptr() for t in out])
    c_lse = (ctypes.c_void_p * n)(*[(t.data_ptr() if t is not None else None) for t in lse])
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    s = stream if stream is not None else torch.cuda.current_stream()
    st = attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), n, ctypes.addressof(c_modes),
                       ctypes.addressof(c_out), ctypes.addressof(c_lse), B, H, Nq, Nk, d, sc, int(chunk_bh),
                       workspace.data_ptr(), workspace.numel(), s.cuda_stream)
    _raise(st, "attn_fwd_host")
    if synchronize:
        s.synchronize()
    return out, lse


def fwd_fp8(q8, k8, v8, descales, causal=False, scale=None, out=None, lse=None, return_lse=True, stream=None):
    """e4m3fn [B,H,N,d] with per-tensor descales (q, k, v) -> (o bf16, lse fp32)."""
    torch = _torch()
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    _check(q8, "q8", torch.float8_e4m3fn)
    _check(k8, "k8", torch.float8_e4m3fn, (B, H, Nk, d))
    _check(v8, "v8", torch.float8_e4m3fn, (B, H, Nk, d))
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q8.device)
    _check(out, "out", torch.bfloat16, (B, H, Nq, d))
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device)
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, H, Nq))
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    dq, dk, dv = (float(x) for x in descales)
    st = attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), dq, dk, dv, out.data_ptr(),
                      lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, sc, int(bool(causal)),
                      _stream(stream))
    _raise(st, "attn_fwd_fp8")
    return out, lse


def paged_decode(q, k_cache, v_cache, block_table, seq_lens, scale=None, out=None, lse=None, workspace=None,
                 return_lse=True, stream=None):
    """q bf16 [B,H,d]; caches bf16 [num_pages, page_size, H, d]; block_table int32
    [B, max_pages]; seq_lens int32 [B] -> (o bf16 [B,H,d], lse fp32 [B,H])."""
    torch = _torch()
    B, H, d = q.shape
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    max_pages = block_table.shape[1]
    _check(q, "q", torch.bfloat16)
    _check(k_cache, "k_cache", torch.bfloat16, (num_pages, page_size, H, d))
    _check(v_cache, "v_cache", torch.bfloat16, (num_pages, page_size, H, d))
    _check(block_table, "block_table", torch.int32, (B, max_pages))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, (B, H, d))
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32, (B, H))
    ws_bytes = attn_paged_decode_workspace_size(B, H, d, max_pages, page_size)
    if ws_bytes == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "attn_paged_decode_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    st = attn_paged_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
                           seq_lens.data_ptr(), B, H, d, page_size, max_pages, num_pages, sc, out.data_ptr(),
                           lse.data_ptr() if lse is not None else None, workspace.data_ptr(), workspace.numel(),
                           _stream(stream))
    _raise(st, "attn_paged_decode")
    return out, lse


def paged_fwd(q, k_cache, v_cache, block_table, seq_lens, cu_seqlens_q=None, max_q_len=None, causal=False,
              scale=None, out=None, lse=None, workspace=None, return_lse=True, stream=None):
    """Tensor-core attention over a paged cache with grouped KV heads.

    q bf16 [total_q, H, d] token-major; caches bf16 [num_pages, page_size,
    H_kv, d]; block_table int32 [B, max_pages]; seq_lens int32 [B];
    cu_seqlens_q int32 [B+1] (None: one query token per request, q [B, H, d]).
    max_q_len is the largest per-request token count (read from
    cu_seqlens_q, with a device-to-host copy, when not given).
    Returns (o bf16 like q, lse fp32 [total_q, H]).
    """
    torch = _torch()
    total_q, H, d = q.shape
    num_pages, page_size, H_kv = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    B, max_pages = block_table.shape
    _check(q, "q", torch.bfloat16)
    _check(k_cache, "k_cache", torch.bfloat16, (num_pages, page_size, H_kv, d))
    _check(v_cache, "v_cache", torch.bfloat16, (num_pages, page_size, H_kv, d))
    _check(block_table, "block_table", torch.int32, (B, max_pages))
    _check(seq_lens, "seq_lens", torch.int32, (B,))
    if cu_seqlens_q is not None:
        _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, (B + 1,))
        if max_q_len is None:
            max_q_len = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B else 0
    else:
        max_q_len = 1
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, (total_q, H, d))
    if lse is None and return_lse:
        lse = torch.empty((total_q, H), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32, (total_q, H))
    ws_bytes = attn_paged_fwd_workspace_size(B, total_q, max_q_len, H, H_kv, d, page_size, max_pages)
    if ws_bytes == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "attn_paged_fwd_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    st = attn_paged_fwd(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
                        cu_seqlens_q.data_ptr() if cu_seqlens_q is not None else None, seq_lens.data_ptr(), B,
                        total_q, max_q_len, H, H_kv, d, page_size, max_pages, num_pages, sc, int(bool(causal)),
                        out.data_ptr(), lse.data_ptr() if lse is not None else None, workspace.data_ptr(),
                        workspace.numel(), _stream(stream))
    _raise(st, "attn_paged_fwd")
    return out, lse


def varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_q_len=None, max_k_len=None, causal=False, scale=None,
               out=None, lse=None, workspace=None, return_lse=True, stream=None):
    """Variable-length batch prefill with grouped KV heads.

    q bf16 [total_q, H, d]; k, v bf16 [total_k, H_kv, d]; cu_seqlens_q,
    cu_seqlens_k int32 [B+1] row offsets.  max_q_len / max_k_len are the
    largest per-request counts (read from the offsets, with a device-to-host
    copy, when not given).  Returns (o bf16 like q, lse fp32 [total_q, H]).
    """
    torch = _torch()
    total_q, H, d = q.shape
    total_k, H_kv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.shape[0] - 1
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (total_k, H_kv, d))
    _check(v, "v", torch.bfloat16, (total_k, H_kv, d))
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, (B + 1,))
    _check(cu_seqlens_k, "cu_seqlens_k", torch.int32, (B + 1,))
    if max_q_len is None:
        max_q_len = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B else 0
    if max_k_len is None:
        max_k_len = int((cu_seqlens_k[1:] - cu_seqlens_k[:-1]).max().item()) if B else 0
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, (total_q, H, d))
    if lse is None and return_lse:
        lse = torch.empty((total_q, H), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32, (total_q, H))
    ws_bytes = attn_varlen_fwd_workspace_size(B, total_q, max_q_len, max_k_len, H, H_kv, d)
    if ws_bytes == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "attn_varlen_fwd_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    st = attn_varlen_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                         B, total_q, total_k, max_q_len, max_k_len, H, H_kv, d, sc, int(bool(causal)), out.data_ptr(),
                         lse.data_ptr() if lse is not None else None, workspace.data_ptr(), workspace.numel(),
                         _stream(stream))
    _raise(st, "attn_varlen_fwd")
    return out, lse


def bwd(q, k, v, o, lse, dout, causal=False, scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients of fwd: (dq, dk, dv) bf16 for the upstream gradient dout, from
    the forward inputs q, k, v, its output o and its lse (same scale and
    causal flag)."""
    torch = _torch()
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check(q, "q", torch.bfloat16)
    _check(k, "k", torch.bfloat16, (B, H, Nk, d))
    _check(v, "v", torch.bfloat16, (B, H, Nk, d))
    _check(o, "o", torch.bfloat16, (B, H, Nq, d))
    _check(dout, "dout", torch.bfloat16, (B, H, Nq, d))
    _check(lse, "lse", torch.float32, (B, H, Nq))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(dq, "dq", torch.bfloat16, q.shape)
    _check(dk, "dk", torch.bfloat16, k.shape)
    _check(dv, "dv", torch.bfloat16, v.shape)
    ws_bytes = attn_bwd_workspace_size(B, H, Nq, d)
    if ws_bytes == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "attn_bwd_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", torch.uint8)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    st = attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, sc, int(bool(causal)),
                  workspace.data_ptr(), workspace.numel(), _stream(stream))
    _raise(st, "attn_bwd")
    return dq, dk, dv


def device_status(stream=None):
    """Synchronise and raise AttnError if a kernel flagged a timeout or bad device data."""
    _raise(attn_device_status(_stream(stream)), "attn_device_status")
