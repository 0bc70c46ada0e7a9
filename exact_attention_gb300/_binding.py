"""ctypes binding of libfa (include/fa.h): argument marshalling only.

The functions named like the C entry points take the same arguments in the
same order; pointer arguments may be ints (device addresses) or torch tensors
(their ``data_ptr()``), ``stream`` may be an int, a ``torch.cuda.Stream`` or
None (the current torch stream). They return the fa_status code as an int.

The tensor-level helpers ``forward``, ``backward`` and ``decode`` allocate the
outputs with torch, call the C entry point and raise :class:`FAError` on any
status other than FA_OK. Every step of the computation runs in the library's
CUDA kernels; there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_F32, FA_F16, FA_BF16 = 0, 1, 2
FA_SCHED_FWD_SPLIT, FA_SCHED_BWD_SPLIT, FA_SCHED_HOST_CHUNKS, FA_SCHED_BWD_PAIR = 1, 2, 3, 4

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

# every symbol include/fa.h declares
EXPORTS = (
    "fa_fwd",
    "fa_fwd_ws",
    "fa_fwd_workspace_bytes",
    "fa_fwd_host",
    "fa_fwd_host_workspace_bytes",
    "fa_fwd_fp8",
    "fa_fwd_fp8_workspace_bytes",
    "fa_bwd",
    "fa_bwd_workspace_bytes",
    "fa_bwd_ws",
    "fa_bwd_ws_workspace_bytes",
    "fa_decode",
    "fa_decode_workspace_bytes",
    "fa_decode_static",
    "fa_decode_ex",
    "fa_decode_ex_workspace_bytes",
    "fa_last_status",
    "fa_status_string",
    "fa_last_error_message",
    "fa_set_wait_budget_ns",
    "fa_set_schedule",
    "fa_debug_inject",
    "fa_debug_schedule_choice",
)

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().fa_last_error_message().decode(errors="replace")
        name = lib().fa_status_string(status).decode(errors="replace")
        super().__init__(f"{where}: {name}: {msg}")


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m exact_attention_gb300.build` "
                           "(there is no fallback implementation)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.fa_fwd.restype = st
    L.fa_fwd_ws.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, f, i, i, vp]
    L.fa_fwd_ws.restype = st
    L.fa_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    L.fa_fwd_workspace_bytes.restype = ctypes.c_size_t
    L.fa_bwd.argtypes = [vp] * 10 + [i, i, i, i, i, f, i, i, vp]
    L.fa_bwd.restype = st
    L.fa_decode.argtypes = [vp] * 5 + [i, i, i, i, f, i, i, vp]
    L.fa_decode.restype = st
    L.fa_decode_static.argtypes = [vp] * 4 + [i, i, i, i, f, i, i, vp]
    L.fa_decode_static.restype = st
    L.fa_decode_workspace_bytes.argtypes = [i, i, i, i]
    L.fa_decode_workspace_bytes.restype = ctypes.c_size_t
    L.fa_bwd_ws.argtypes = [vp] * 10 + [ctypes.c_size_t, i, i, i, i, i, f, i, i, vp]
    L.fa_bwd_ws.restype = st
    L.fa_bwd_ws_workspace_bytes.argtypes = [i, i, i, i]
    L.fa_bwd_ws_workspace_bytes.restype = ctypes.c_size_t
    L.fa_fwd_host.argtypes = [vp] * 6 + [ctypes.c_size_t, i, i, i, i, i, f, i, i, vp]
    L.fa_fwd_host.restype = st
    L.fa_fwd_fp8.argtypes = [vp] * 7 + [ctypes.c_size_t, i, i, i, i, i, f, i, i, vp]
    L.fa_fwd_fp8.restype = st
    L.fa_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i, i]
    L.fa_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
    L.fa_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    L.fa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    L.fa_decode_ex.argtypes = [vp] * 6 + [i, i, i, i, i, f, i, i, vp]
    L.fa_decode_ex.restype = st
    L.fa_decode_ex_workspace_bytes.argtypes = [i, i, i, i, i]
    L.fa_decode_ex_workspace_bytes.restype = ctypes.c_size_t
    L.fa_bwd_workspace_bytes.argtypes = [i, i, i]
    L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.fa_last_status.argtypes = [vp]
    L.fa_last_status.restype = st
    L.fa_status_string.argtypes = [st]
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_last_error_message.argtypes = []
    L.fa_last_error_message.restype = ctypes.c_char_p
    L.fa_set_wait_budget_ns.argtypes = [ctypes.c_ulonglong]
    L.fa_set_wait_budget_ns.restype = st
    L.fa_set_schedule.argtypes = [i, i]
    L.fa_set_schedule.restype = st
    L.fa_debug_inject.argtypes = [i]
    L.fa_debug_inject.restype = st
    L.fa_debug_schedule_choice.argtypes = [i] * 7
    L.fa_debug_schedule_choice.restype = i
    _lib = L
    return L


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------- C entry points
def fa_fwd(Q, K, V, O, LSE, B, H, M, N, D, scale, causal, dtype, stream=None) -> int:
    return lib().fa_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, M, N, D, float(scale), int(causal),
                        int(dtype), _stream(stream))

def fa_fwd_ws(Q, K, V, O, LSE, workspace, workspace_bytes, B, H, M, N, D, scale, causal, dtype, stream=None) -> int:
    return lib().fa_fwd_ws(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(workspace), int(workspace_bytes), B, H,
                           M, N, D, float(scale), int(causal), int(dtype), _stream(stream))


def fa_fwd_workspace_bytes(B, H, M, N, D, causal, dtype) -> int:
    return lib().fa_fwd_workspace_bytes(B, H, M, N, D, int(causal), int(dtype))


def fa_bwd_ws(Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, B, H, M, N, D, scale, causal, dtype,
              stream=None) -> int:
    return lib().fa_bwd_ws(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(dK), _ptr(dV),
                           _ptr(workspace), workspace_bytes, B, H, M, N, D, float(scale), int(causal), int(dtype),
                           _stream(stream))


def fa_bwd_ws_workspace_bytes(B, H, M, D) -> int:
    return lib().fa_bwd_ws_workspace_bytes(B, H, M, D)


def fa_fwd_host(hQ, hK, hV, hO, hLSE, dev_ws, dev_ws_bytes, B, H, M, N, D, scale, causal, dtype, stream=None) -> int:
    return lib().fa_fwd_host(_ptr(hQ), _ptr(hK), _ptr(hV), _ptr(hO), _ptr(hLSE), _ptr(dev_ws), dev_ws_bytes, B, H, M,
                             N, D, float(scale), int(causal), int(dtype), _stream(stream))


def fa_fwd_host_workspace_bytes(B, H, M, N, D, causal, dtype) -> int:
    return lib().fa_fwd_host_workspace_bytes(B, H, M, N, D, int(causal), int(dtype))


def fa_fwd_fp8(Q, K, V, O, LSE, signs, workspace, workspace_bytes, B, H, M, N, D, scale, causal, dtype,
               stream=None) -> int:
    return lib().fa_fwd_fp8(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(signs), _ptr(workspace),
                            int(workspace_bytes), B, H, M, N, D, float(scale), int(causal), int(dtype),
                            _stream(stream))


def fa_fwd_fp8_workspace_bytes(B, H, M, N, D) -> int:
    return lib().fa_fwd_fp8_workspace_bytes(B, H, M, N, D)



def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, delta_ws, B, H, M, N, D, scale, causal, dtype, stream=None) -> int:
    return lib().fa_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ), _ptr(dK), _ptr(dV),
                        _ptr(delta_ws), B, H, M, N, D, float(scale), int(causal), int(dtype), _stream(stream))


def fa_decode(q, Kcache, Vcache, O, partial_ws, B, H, N, D, scale, n_splits, dtype, stream=None) -> int:
    return lib().fa_decode(_ptr(q), _ptr(Kcache), _ptr(Vcache), _ptr(O), _ptr(partial_ws), B, H, N, D,
                           float(scale), int(n_splits), int(dtype), _stream(stream))


def fa_decode_static(q, Kcache, Vcache, O, B, H, N, D, scale, n_splits, dtype, stream=None) -> int:
    """Decode with the library's own fixed scratch (no workspace, no allocation); see include/fa.h."""
    return lib().fa_decode_static(_ptr(q), _ptr(Kcache), _ptr(Vcache), _ptr(O), B, H, N, D, float(scale),
                                  int(n_splits), int(dtype), _stream(stream))


def fa_decode_workspace_bytes(B, H, D, n_splits) -> int:
    return lib().fa_decode_workspace_bytes(B, H, D, n_splits)


def fa_decode_ex(q, Kcache, Vcache, O, LSE, partial_ws, B, H, R, N, D, scale, n_splits, dtype, stream=None) -> int:
    return lib().fa_decode_ex(_ptr(q), _ptr(Kcache), _ptr(Vcache), _ptr(O), _ptr(LSE), _ptr(partial_ws), B, H, R, N,
                              D, float(scale), n_splits, int(dtype), _stream(stream))


def fa_decode_ex_workspace_bytes(B, H, R, D, n_splits) -> int:
    return lib().fa_decode_ex_workspace_bytes(B, H, R, D, n_splits)


def fa_bwd_workspace_bytes(B, H, M) -> int:
    return lib().fa_bwd_workspace_bytes(B, H, M)


def fa_last_status(stream=None) -> int:
    return lib().fa_last_status(_stream(stream))


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(status).decode()


def fa_last_error_message() -> str:
    return lib().fa_last_error_message().decode(errors="replace")


def fa_set_wait_budget_ns(ns: int) -> int:
    return lib().fa_set_wait_budget_ns(int(ns))

def fa_set_schedule(key: int, value: int) -> int:
    return lib().fa_set_schedule(int(key), int(value))


class schedule:
    """Context manager: fa_set_schedule(key, value) inside the block, automatic (-1) after it."""

    def __init__(self, key: int, value: int):
        self.key, self.value = key, value

    def __enter__(self):
        _check(fa_set_schedule(self.key, self.value), "fa_set_schedule")
        return self

    def __exit__(self, *exc):
        fa_set_schedule(self.key, -1)
        return False


def fa_debug_inject(kind: int) -> int:
    return lib().fa_debug_inject(int(kind))


def fa_debug_schedule_choice(which: int, B: int, H: int, M: int, N: int, causal: bool, num_sms: int) -> int:
    return lib().fa_debug_schedule_choice(int(which), B, H, M, N, int(causal), num_sms)



# ------------------------------------------------------- tensor helpers
def fa_dtype(t) -> int:
    import torch
    m = {torch.float32: FA_F32, torch.float16: FA_F16, torch.bfloat16: FA_BF16}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _check(status: int, where: str):
    if status != FA_OK:
        raise FAError(status, where)


def _dims4(t, name):
    if t.dim() != 4 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor [B, H, rows, D]")
    return t.shape


_fwd_workspaces = {}  # device index -> zero-filled uint8 tensor (grown on demand)


def forward_workspace(device, nbytes: int):
    """A zero-filled device buffer of at least nbytes for fa_fwd_ws, kept per device and
    reused by later calls (they run in stream order on one stream; two streams calling
    forward at once would need a workspace each)."""
    import torch
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    ws = _fwd_workspaces.get(idx)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=f"cuda:{idx}")
        _fwd_workspaces[idx] = ws
    return ws


def forward(q, k, v, scale: float, causal: bool = False, out=None, lse=None, stream=None, workspace=None):
    """O, LSE = attention(q [B,H,M,D], k/v [B,H,N,D]); LSE is float32 [B,H,M].

    workspace: None uses a cached per-device workspace (see forward_workspace); False
    runs without one (fa_fwd); a zero-initialised uint8 tensor is used as given."""
    import torch
    B, H, M, D = _dims4(q, "q")
    N = _dims4(k, "k")[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    dt = fa_dtype(q)
    nbytes = fa_fwd_workspace_bytes(B, H, M, N, D, causal, dt) if workspace is not False else 0
    if nbytes == 0:
        _check(fa_fwd(q, k, v, out, lse, B, H, M, N, D, scale, causal, dt, stream), "fa_fwd")
        return out, lse
    ws = forward_workspace(q.device, nbytes) if workspace is None else workspace
    _check(fa_fwd_ws(q, k, v, out, lse, ws, ws.numel() * ws.element_size(), B, H, M, N, D, scale, causal, dt, stream),
           "fa_fwd_ws")
    return out, lse


def forward_fp8(q, k, v, scale: float, causal: bool, signs, out=None, lse=None, workspace=None, stream=None):
    """O, LSE of the FP8 forward (D = 64); signs: a device int8 tensor of 64 entries +-1. Returns
    (O, LSE, workspace); the workspace holds the E4M3 operands and their scales afterwards."""
    import torch
    B, H, M, D = _dims4(q, "q")
    N = _dims4(k, "k")[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    nbytes = fa_fwd_fp8_workspace_bytes(B, H, M, N, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _check(fa_fwd_fp8(q, k, v, out, lse, signs, workspace, workspace.numel(), B, H, M, N, D, scale, causal,
                      fa_dtype(q), stream), "fa_fwd_fp8")
    return out, lse, workspace


def backward(q, k, v, o, do, lse, scale: float, causal: bool = False, stream=None, fused: bool = True):
    """dQ, dK, dV of sum(do * o); also returns delta (rowsum(dO o O)).

    fused=True (default) goes through fa_bwd_ws (one dK/dV/dQ pass for D = 64, with an f32 dQ
    accumulator in the same workspace after delta); fused=False through fa_bwd (the three kernels:
    delta, dK/dV, dQ)."""
    import torch
    B, H, M, D = _dims4(q, "q")
    N = _dims4(k, "k")[2]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if fused:
        nbytes = fa_bwd_ws_workspace_bytes(B, H, M, D)
        ws = torch.empty((max(nbytes, 4) // 4,), dtype=torch.float32, device=q.device)
        _check(fa_bwd_ws(q, k, v, o, do, lse, dq, dk, dv, ws, nbytes, B, H, M, N, D, scale, causal, fa_dtype(q),
                         stream), "fa_bwd_ws")
        return dq, dk, dv, ws[: B * H * M].view(B, H, M)
    ws = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    _check(fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, B, H, M, N, D, scale, causal, fa_dtype(q), stream),
           "fa_bwd")
    return dq, dk, dv, ws


def decode(q, k_cache, v_cache, scale: float, n_splits: int, out=None, workspace=None, stream=None, lse=None):
    """O [B,H,R,D] for R (1..4) query rows per (batch, head); returns (O, partial workspace).

    With lse (a float32 [B,H,R] tensor, or True to allocate one) the LSE is written too and
    (O, workspace, lse) is returned; R = 1 without lse goes through fa_decode."""
    import torch
    B, H, R, D = _dims4(q, "q")
    N = _dims4(k_cache, "k_cache")[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is True:
        lse = torch.empty((B, H, R), dtype=torch.float32, device=q.device)
    if R == 1 and lse is None:
        if workspace is None:
            nbytes = fa_decode_workspace_bytes(B, H, D, n_splits)
            workspace = torch.empty((max(nbytes, 4) // 4,), dtype=torch.float32, device=q.device)
        _check(fa_decode(q, k_cache, v_cache, out, workspace, B, H, N, D, scale, n_splits, fa_dtype(q), stream),
               "fa_decode")
        return out, workspace
    if workspace is None:
        nbytes = fa_decode_ex_workspace_bytes(B, H, R, D, n_splits)
        workspace = torch.empty((max(nbytes, 4) // 4,), dtype=torch.float32, device=q.device)
    _check(fa_decode_ex(q, k_cache, v_cache, out, lse, workspace, B, H, R, N, D, scale, n_splits, fa_dtype(q),
                        stream), "fa_decode_ex")
    return (out, workspace) if lse is None else (out, workspace, lse)


def split_workspace(ws, B: int, H: int, D: int, n_splits: int):
    """Views (O_s [B*H, n_splits, D], m_s [B*H, n_splits], l_s [B*H, n_splits]) of a decode workspace."""
    BH = B * H
    o = ws[: BH * n_splits * D].view(BH, n_splits, D)
    m = ws[BH * n_splits * D: BH * n_splits * (D + 1)].view(BH, n_splits)
    l_ = ws[BH * n_splits * (D + 1): BH * n_splits * (D + 2)].view(BH, n_splits)
    return o, m, l_
