"""ctypes wrapper of the fp64 CPU oracle (``gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg use it. The CUDA library never imports, links or calls it, and it
shares no code with the CUDA library.

Every function takes and returns numpy float64 arrays; inputs given in bf16 or
fp32 are promoted exactly (bf16 -> fp64 and fp32 -> fp64 are exact).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_DIR = Path(__file__).resolve().parent
_SRC = _DIR / "gdn_oracle.c"
_SO = _DIR / "_build" / "libgdn_oracle.so"
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> Path:
    """Compile the oracle with gcc (ISO C99: no FMA contraction, plain IEEE fp64)."""
    if force or not _SO.exists() or _SO.stat().st_mtime < _SRC.stat().st_mtime:
        _SO.parent.mkdir(parents=True, exist_ok=True)
        tmp = _SO.with_suffix(f".{os.getpid()}.tmp")
        subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-pthread",
                        str(_SRC), "-o", str(tmp), "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        lib.gdn_oracle_layer.restype = ctypes.c_int
        lib.gdn_oracle_mask_length.restype = ctypes.c_int
        for name in ("gdn_oracle_gates", "gdn_oracle_conv", "gdn_oracle_l2norm",
                     "gdn_oracle_recurrence", "gdn_oracle_gated_rmsnorm"):
            getattr(lib, name).restype = None
        _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact promotion to a C-contiguous float64 array (accepts torch tensors)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_dp)


def gates(a, b, A_log, dt_bias, mask=None):
    """g, beta for one row: a, b [T, nv]; mask [T] or None. Returns (g, beta)."""
    a, b, A_log, dt_bias = map(_f64, (a, b, A_log, dt_bias))
    T, nv = a.shape
    m = _f64(mask) if mask is not None else None
    g = np.empty((T, nv)); beta = np.empty((T, nv))
    _load().gdn_oracle_gates(T, nv, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(m), _p(g), _p(beta))
    return g, beta


def conv(x, w, conv_state, Lr=None, ckpt=False):
    """Depthwise causal conv + SiLU continued from ``conv_state``.

    x [T, C], w [C, K], conv_state [K-1, C]. Returns (y [T, C], new_tail [K-1, C],
    tail_ckpt [T, K-1, C] or None)."""
    x, w = _f64(x), _f64(w)
    st = _f64(conv_state).copy()
    T, C = x.shape
    K = w.shape[1]
    Lr = T if Lr is None else int(Lr)
    y = np.empty((T, C))
    ck = np.empty((T, K - 1, C)) if ckpt else None
    _load().gdn_oracle_conv(T, C, K, _p(x), _p(w), _p(st), Lr, _p(y), _p(ck))
    return y, st, ck


def l2norm(x, eps=1e-6, scale=1.0):
    x = _f64(x)
    out = np.empty_like(x)
    _load().gdn_oracle_l2norm(x.size, _p(x), ctypes.c_double(eps), ctypes.c_double(scale), _p(out))
    return out


def recurrence(q, k, v, g, beta, S, ckpt=False):
    """Token-by-token gated delta rule for one head on the stored transpose
    S [dk, dv]. q, k [T, dk] (normalised), v [T, dv], g, beta [T].
    Returns (o [T, dv], S_final [dk, dv], ckpt [T, dk, dv] or None)."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    S = _f64(S).copy()
    T, dk = q.shape
    dv = v.shape[1]
    o = np.empty((T, dv))
    ck = np.empty((T, dk, dv)) if ckpt else None
    _load().gdn_oracle_recurrence(T, dk, dv, _p(q), _p(k), _p(v), _p(g), _p(beta), _p(S), _p(o), _p(ck))
    return o, S, ck


def gated_rmsnorm(o, z, w, eps=1e-6):
    o, z, w = map(_f64, (o, z, w))
    out = np.empty_like(o)
    _load().gdn_oracle_gated_rmsnorm(o.size, _p(o), _p(z), _p(w), ctypes.c_double(eps), _p(out))
    return out


def mask_length(mask) -> int:
    m = _f64(mask)
    return _load().gdn_oracle_mask_length(m.size, _p(m))


def layer(*, q, k, v, z, a, b, A_log, dt_bias, conv_w, norm_w, conv_state, state,
          nk, nv, dk, dv, mask=None, scale=None, l2_eps=1e-6, rms_eps=1e-6,
          checkpoints=False, n_threads=None):
    """One Gated DeltaNet layer over B rows of T tokens (dense layout).

    q, k [B, T, nk*dk]; v, z [B, T, nv*dv]; a, b [B, T, nv]; A_log, dt_bias [nv];
    conv_w [C, K]; norm_w [dv]; conv_state [B, K-1, C]; state [B, nv, dk, dv];
    mask [B, T] or None.  Inputs are not modified.

    Returns a dict: out [B, T, nv, dv], conv_state, state, and, when
    ``checkpoints`` is set, ckpt_state [B, T, nv, dk, dv] and
    ckpt_conv [B, T, K-1, C]."""
    q, k, v, z, a, b = map(_f64, (q, k, v, z, a, b))
    A_log, dt_bias, conv_w, norm_w = map(_f64, (A_log, dt_bias, conv_w, norm_w))
    cs = _f64(conv_state).copy()
    st = _f64(state).copy()
    B, T = q.shape[0], q.shape[1]
    K = conv_w.shape[1]
    C = 2 * nk * dk + nv * dv
    m = _f64(mask) if mask is not None else None
    if scale is None:
        scale = dk ** -0.5
    out = np.zeros((B, T, nv * dv))
    cks = np.empty((B, T, nv, dk, dv)) if checkpoints else None
    ckc = np.empty((B, T, K - 1, C)) if checkpoints else None
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    rc = _load().gdn_oracle_layer(
        B, T, nk, nv, dk, dv, K, ctypes.c_double(scale), ctypes.c_double(l2_eps),
        ctypes.c_double(rms_eps), _p(q), _p(k), _p(v), _p(z), _p(a), _p(b), _p(A_log),
        _p(dt_bias), _p(conv_w), _p(norm_w), _p(m), _p(cs), _p(st), _p(out), _p(cks), _p(ckc),
        int(n_threads))
    if rc != 0:
        raise ValueError("mask rows must be a prefix of ones followed by zeros")
    res = {"out": out.reshape(B, T, nv, dv), "conv_state": cs, "state": st}
    if checkpoints:
        res["ckpt_state"] = cks
        res["ckpt_conv"] = ckc
    return res


def in_proj(hidden, w_in, nk, nv, dk, dv):
    """The layer's in-projection and its split (statecache.py, CacheQwen35._gdn:
    the features of hidden x in_proj^T in the order [mixed (2 kd + vd), z (vd),
    b (nv), a (nv)], mixed = [q (kd), k (kd), v (vd)]). hidden [M, H], w_in [N, H].
    Returns the six float64 arrays, each [M, width]. The product is numpy's fp64
    matmul of the exact inputs."""
    x, w = _f64(hidden), _f64(w_in)
    y = x.reshape(-1, x.shape[-1]) @ w.T
    kd, vd = nk * dk, nv * dv
    cuts = np.cumsum([kd, kd, vd, vd, nv])
    q, k, v, z, b, a = np.split(y, cuts, axis=1)
    return {"q": q, "k": k, "v": v, "z": z, "b": b, "a": a}


def out_proj(o, w_out):
    """The layer's out-projection: o [M, V] x w_out [H, V]^T in fp64."""
    x, w = _f64(o), _f64(w_out)
    return x.reshape(-1, x.shape[-1]) @ w.T
