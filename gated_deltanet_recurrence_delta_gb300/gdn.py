"""Thin ctypes binding of ``libgdn.so`` (the C-ABI declared in ``include/gdn.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (device memory and streams come from
PyTorch); their data pointers are handed to the C entry points of the same
names. A non-OK status raises :class:`GdnError`. If the library has not been
built, the first call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_build" / "libgdn.so"

STATUS = {0: "GDN_OK", 1: "GDN_ERR_ARG", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_MASK", 4: "GDN_ERR_INDEX",
          5: "GDN_ERR_CUDA", 6: "GDN_ERR_WORKSPACE", 7: "GDN_ERR_TIMEOUT"}
EXPORTS = ("gdn_decode_step", "gdn_verify_with_checkpoints", "gdn_prefill_chunked",
           "gdn_prefill_workspace_size", "gdn_state_copy", "gdn_check_status", "gdn_last_error",
           "gdn_prefill_chunked_static_scratch", "gdn_commit_accepted", "gdn_decode_step_mxfp8",
           "gdn_prefill_chunked_ckpt", "gdn_in_proj", "gdn_out_proj", "gdn_copy_overlapped")
MAX_OVERLAPPED_COPIES = 8


class GdnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code
        self.name = STATUS.get(code, str(code))


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "T", "nk", "nv", "dk", "dv", "conv_k", "n_slots")] + [
        ("scale", ctypes.c_float), ("l2_eps", ctypes.c_float), ("rms_eps", ctypes.c_float)]


class Inputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "z", "a", "b", "A_log", "dt_bias", "conv_w",
                                               "norm_w", "mask", "cu_seqlens", "state_idx")]


class InputsMxfp8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "z", "q_scale", "k_scale", "v_scale", "z_scale", "a",
                                               "b", "A_log", "dt_bias", "conv_w", "norm_w", "mask", "state_idx")]


class Copy(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


_lib = None


def load_library(path: Path | str | None = None):
    """Load libgdn.so (in-tree build). Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise RuntimeError(f"{p} is not built; run gated_deltanet_recurrence_delta_gb300.build.build()")
    lib = ctypes.CDLL(str(p))
    P = ctypes.c_void_p
    DP = ctypes.POINTER(Dims)
    IP = ctypes.POINTER(Inputs)
    lib.gdn_decode_step.argtypes = [DP, IP, P, P, P, P]
    lib.gdn_verify_with_checkpoints.argtypes = [DP, IP, P, P, P, P, P, P]
    lib.gdn_prefill_chunked.argtypes = [DP, IP, P, P, P, P, ctypes.c_size_t, P]
    lib.gdn_prefill_chunked_static_scratch.argtypes = [DP, IP, P, P, P, P]
    lib.gdn_prefill_workspace_size.argtypes = [DP, ctypes.c_int]
    lib.gdn_prefill_workspace_size.restype = ctypes.c_size_t
    lib.gdn_state_copy.argtypes = [DP, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P]
    lib.gdn_prefill_chunked_ckpt.argtypes = [DP, IP, P, P, P, P, ctypes.c_size_t, P, ctypes.c_int32, P, P,
                                             ctypes.c_int32, P]
    lib.gdn_in_proj.argtypes = [DP, ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P, P, P, P]
    lib.gdn_out_proj.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P, P]
    lib.gdn_decode_step_mxfp8.argtypes = [DP, ctypes.POINTER(InputsMxfp8), P, P, P, P]
    lib.gdn_commit_accepted.argtypes = [DP, ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P, P, P]
    lib.gdn_copy_overlapped.argtypes = [ctypes.POINTER(Copy), ctypes.c_int32, P]
    lib.gdn_check_status.argtypes = [P]
    lib.gdn_last_error.restype = ctypes.c_char_p
    for name in ("gdn_decode_step", "gdn_verify_with_checkpoints", "gdn_prefill_chunked", "gdn_state_copy",
                 "gdn_check_status", "gdn_prefill_chunked_static_scratch", "gdn_commit_accepted",
                 "gdn_decode_step_mxfp8", "gdn_prefill_chunked_ckpt", "gdn_in_proj", "gdn_out_proj",
                 "gdn_copy_overlapped"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def last_error() -> str:
    return load_library().gdn_last_error().decode()


def _check(code: int):
    if code != 0:
        raise GdnError(code, last_error())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_dims(B, T, nk, nv, dk, dv, n_slots, conv_k=4, scale=None, l2_eps=1e-6, rms_eps=1e-6) -> Dims:
    return Dims(B=B, T=T, nk=nk, nv=nv, dk=dk, dv=dv, conv_k=conv_k, n_slots=n_slots,
                scale=dk ** -0.5 if scale is None else scale, l2_eps=l2_eps, rms_eps=rms_eps)


def make_inputs(q, k, v, z, a, b, A_log, dt_bias, conv_w, norm_w, mask=None, cu_seqlens=None,
                state_idx=None) -> Inputs:
    """The inputs struct of raw device pointers. It keeps references to the
    tensors, so they (and their device memory) live as long as the struct."""
    inp = Inputs(q=_ptr(q), k=_ptr(k), v=_ptr(v), z=_ptr(z), a=_ptr(a), b=_ptr(b), A_log=_ptr(A_log),
                 dt_bias=_ptr(dt_bias), conv_w=_ptr(conv_w), norm_w=_ptr(norm_w), mask=_ptr(mask),
                 cu_seqlens=_ptr(cu_seqlens), state_idx=_ptr(state_idx))
    inp._tensors = (q, k, v, z, a, b, A_log, dt_bias, conv_w, norm_w, mask, cu_seqlens, state_idx)
    return inp


def make_inputs_mxfp8(q, k, v, z, q_scale, k_scale, v_scale, z_scale, a, b, A_log, dt_bias, conv_w, norm_w,
                      mask=None, state_idx=None) -> InputsMxfp8:
    """The MXFP8 inputs struct (e4m3 q/k/v/z as uint8 tensors, their E8M0
    block scales as uint8 tensors); keeps references to the tensors."""
    t = (q, k, v, z, q_scale, k_scale, v_scale, z_scale, a, b, A_log, dt_bias, conv_w, norm_w, mask, state_idx)
    inp = InputsMxfp8(*(_ptr(x) for x in t))
    inp._tensors = t
    return inp


def decode_step_mxfp8(dims: Dims, inputs: InputsMxfp8, conv_state, recurrent_state, out, stream=None):
    _check(load_library().gdn_decode_step_mxfp8(ctypes.byref(dims), ctypes.byref(inputs), _ptr(conv_state),
                                                _ptr(recurrent_state), _ptr(out), _stream(stream)))


def copy_overlapped(copies, stream=None):
    """gdn_copy_overlapped: up to MAX_OVERLAPPED_COPIES copies given as
    (dst, src, nbytes) -- tensors or raw addresses, device memory or pinned
    host memory -- done by one kernel that runs alongside the kernel before it
    on the stream and completes after it. The caller keeps the buffers alive
    and untouched until the stream has passed the call."""
    arr = (Copy * max(1, len(copies)))(*[Copy(_ptr(d), _ptr(s), int(n)) for d, s, n in copies])
    _check(load_library().gdn_copy_overlapped(arr, len(copies), _stream(stream)))


def decode_step(dims: Dims, inputs: Inputs, conv_state, recurrent_state, out, stream=None):
    _check(load_library().gdn_decode_step(ctypes.byref(dims), ctypes.byref(inputs), _ptr(conv_state),
                                          _ptr(recurrent_state), _ptr(out), _stream(stream)))


def verify_with_checkpoints(dims: Dims, inputs: Inputs, conv_state, recurrent_state, out, ckpt_state, ckpt_conv,
                            stream=None):
    _check(load_library().gdn_verify_with_checkpoints(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(conv_state), _ptr(recurrent_state), _ptr(out),
        _ptr(ckpt_state), _ptr(ckpt_conv), _stream(stream)))


def prefill_workspace_size(dims: Dims, packed: bool = False) -> int:
    """Workspace bytes of a prefill call: dense rows, or packed rows (cu_seqlens)."""
    return int(load_library().gdn_prefill_workspace_size(ctypes.byref(dims), int(bool(packed))))


def prefill_chunked(dims: Dims, inputs: Inputs, conv_state, recurrent_state, out, workspace, workspace_bytes=None,
                    stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load_library().gdn_prefill_chunked(ctypes.byref(dims), ctypes.byref(inputs), _ptr(conv_state),
                                              _ptr(recurrent_state), _ptr(out), _ptr(workspace),
                                              int(workspace_bytes), _stream(stream)))


def prefill_chunked_ckpt(dims: Dims, inputs: Inputs, conv_state, recurrent_state, out, workspace, ckpt, ckpt_state,
                         ckpt_conv, workspace_bytes=None, stream=None):
    """gdn_prefill_chunked_ckpt: ckpt is a device int32 [n, 3] tensor of (row,
    position, slot); ckpt_state / ckpt_conv the checkpoint slots."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    n = 0 if ckpt is None else int(ckpt.shape[0])
    _check(load_library().gdn_prefill_chunked_ckpt(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(conv_state), _ptr(recurrent_state), _ptr(out),
        _ptr(workspace), int(workspace_bytes), _ptr(ckpt), n, _ptr(ckpt_state), _ptr(ckpt_conv),
        int(ckpt_state.shape[0]) if ckpt_state is not None else 0, _stream(stream)))


def prefill_chunked_static_scratch(dims: Dims, inputs: Inputs, conv_state, recurrent_state, out, stream=None):
    """gdn_prefill_chunked with the library's own 64 MiB static scratch (for
    callers that cannot allocate device memory)."""
    _check(load_library().gdn_prefill_chunked_static_scratch(ctypes.byref(dims), ctypes.byref(inputs),
                                                             _ptr(conv_state), _ptr(recurrent_state), _ptr(out),
                                                             _stream(stream)))


def state_copy(dims: Dims, src_state, src_conv, dst_state, dst_conv, src_slot, dst_slot, n, n_src_slots,
               n_dst_slots, stream=None):
    _check(load_library().gdn_state_copy(ctypes.byref(dims), _ptr(src_state), _ptr(src_conv), _ptr(dst_state),
                                         _ptr(dst_conv), _ptr(src_slot), _ptr(dst_slot), int(n),
                                         int(n_src_slots), int(n_dst_slots), _stream(stream)))


def commit_accepted(dims: Dims, n_layers, paths, ckpt_state, ckpt_conv, state_pool, conv_pool, accept_len, dst_slot,
                    winner=None, stream=None):
    """gdn_commit_accepted: every layer's winning checkpoint into its pool, one launch."""
    _check(load_library().gdn_commit_accepted(ctypes.byref(dims), int(n_layers), int(paths), _ptr(ckpt_state),
                                              _ptr(ckpt_conv), _ptr(state_pool), _ptr(conv_pool), _ptr(accept_len),
                                              _ptr(dst_slot), _ptr(winner), _stream(stream)))


def commit_source_slot(accept_len, T: int) -> tuple[int, int]:
    """The checkpoint to commit after a verify call of len(accept_len) paths x T
    draft tokens: (winner path, checkpoint slot for gdn_state_copy's src_slot).

    generate.py (sparkle, mlx_streaming/mtp), commit_tree_row(row, accepted_len):
    the winner is the first path with the longest accept length (ties go to the
    lower index); its checkpoint slot is winner * T + L - 1, the state after its
    L accepted tokens. L = 0 commits nothing: slot -1 (gdn_state_copy skips it).
    Host arithmetic only."""
    L = [int(x) for x in accept_len]
    if not L or any(x < 0 or x > T for x in L):
        raise ValueError("accept lengths must lie in [0, T] and there must be at least one path")
    win = max(range(len(L)), key=lambda p: (L[p], -p))
    return win, (win * T + L[win] - 1 if L[win] > 0 else -1)


def in_proj(dims: Dims, hidden, w_in, q, k, v, z, a, b, stream=None):
    """gdn_in_proj: hidden [M, H] x w_in [N, H]^T split into q, k, v, z, a, b."""
    H = int(hidden.shape[-1])
    M = hidden.numel() // H
    _check(load_library().gdn_in_proj(ctypes.byref(dims), M, H, _ptr(hidden), _ptr(w_in), _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(z), _ptr(a), _ptr(b), _stream(stream)))


def out_proj(o, w_out, y, stream=None):
    """gdn_out_proj: y [M, H] = o [M, V] x w_out [H, V]^T."""
    V, H = int(o.shape[-1]), int(w_out.shape[0])
    M = o.numel() // V
    _check(load_library().gdn_out_proj(M, H, V, _ptr(o), _ptr(w_out), _ptr(y), _stream(stream)))


def check_status(stream=None):
    """Synchronise the stream and raise on a device-detected error."""
    _check(load_library().gdn_check_status(_stream(stream)))


def workspace(dims: Dims, packed: bool = False, device="cuda") -> torch.Tensor:
    """A workspace tensor for gdn_prefill_chunked (torch allocations are
    256-byte aligned); packed: the call passes cu_seqlens."""
    n = prefill_workspace_size(dims, packed)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)
