"""The layer's three scalar parameters in gdn_dims -- the query scale, the q/k
L2-norm epsilon and the RMSNorm epsilon -- reach every path, through the C-ABI:
decode, verify with checkpoints, the tensor-core prefill in its one-grid form
(dense rows) and in its separate-kernel form (packed rows), and the CUDA-core
prefill (head size 32), each against the fp64 oracle given the same values.

The values are chosen so that each one moves the result far past the bars:
with scale = 1 the outputs o grow by ~11x, which the gated RMSNorm cancels
except through its epsilon, set to 1e-2, about mean(o^2) at that scale; the
L2-norm epsilon of 2 shortens the normalised q and k by a few percent, which
moves the state. Each test first checks, on the oracle alone, that putting any
one of the three back to its default changes the reference by more than ten
times the bars: a path that ignored one of them would fail."""
import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from tests.gpu_cases import (ACTS, OUT_ATOL, STATE_RTOL, WEIGHTS, assert_out, assert_state, dev, dims, inputs,
                             max_abs, oracle_layer, rel_fro)

pytestmark = pytest.mark.gpu

PARAMS = dict(scale=1.0, l2_eps=2.0, rms_eps=1e-2)
DEFAULTS = dict(scale=None, l2_eps=1e-6, rms_eps=1e-6)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    build.build()
    gdn.load_library()


def _wd(d):
    return {n: dev(d[n]) for n in WEIGHTS}


def _reference(oracle_mod, shape, d, acts, conv, state, mask=None, checkpoints=False, real=None):
    """The oracle with PARAMS, after checking that each parameter alone, put
    back to its default, moves the outputs (at real tokens) and the state by
    more than ten times the bars."""
    ref = oracle_layer(oracle_mod, shape, d, acts, conv, state, mask=mask, checkpoints=checkpoints, **PARAMS)
    for name in PARAMS:
        alt = oracle_layer(oracle_mod, shape, d, acts, conv, state, mask=mask, **{**PARAMS, name: DEFAULTS[name]})
        o, o_alt = ref["out"], alt["out"]
        if real is not None:
            o, o_alt = o[:, :real], o_alt[:, :real]
        moved_out = float(abs(o - o_alt).max())
        moved_state = rel_fro(torch.from_numpy(alt["state"]), ref["state"])
        assert moved_out > 10 * OUT_ATOL or moved_state > 10 * STATE_RTOL, \
            f"{name}: the reference barely moves (out {moved_out:.2e}, state {moved_state:.2e})"
    return ref


@pytest.mark.parametrize("shape", [I.Shape(nk=2, nv=4, dk=128, dv=128), I.TINY])
def test_decode_params(oracle_mod, shape):
    d = I.decode_batch(seed=160, B=3, shape=shape)
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = torch.empty((3, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    gdn.decode_step(dims(shape, 3, 1, 3, **PARAMS), inputs(w, {n: dev(d[n]) for n in ACTS}), conv, S, out)
    gdn.check_status()
    ref = _reference(oracle_mod, shape, d, d, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])


def test_verify_params(oracle_mod):
    shape, B, T = I.Shape(nk=2, nv=4, dk=128, dv=128), 2, 8
    d = I.decode_batch(seed=161, B=B, shape=shape)
    acts = I.activations(shape, B, T, torch.Generator().manual_seed(162))
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = torch.empty((B, T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    ck_s = torch.empty((B, T, shape.nv, shape.dk, shape.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.empty((B, T, 3, shape.C), dtype=torch.bfloat16, device="cuda")
    gdn.verify_with_checkpoints(dims(shape, B, T, B, **PARAMS), inputs(w, {n: dev(a) for n, a in acts.items()}),
                                conv, S, out, ck_s, ck_c)
    gdn.check_status()
    ref = _reference(oracle_mod, shape, d, acts, d["conv_state"], d["state"], checkpoints=True)
    assert_out(out, ref["out"])
    for t in range(T):
        assert_state(ck_s[:, t], ref["ckpt_state"][:, t], f"checkpoint {t}")


def _prefill(shape, w, acts, conv, S, B, T, mask=None, cu=None):
    out = torch.empty((acts["q"].shape[0], T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    dm = dims(shape, B, T, conv.shape[0], **PARAMS)
    ws = gdn.workspace(dm, packed=cu is not None)
    gdn.prefill_chunked(dm, inputs(w, acts, mask=mask, cu=cu), conv, S, out, ws)
    return out


@pytest.mark.parametrize("shape,T", [(I.Shape(nk=2, nv=4, dk=128, dv=128), 130), (I.TINY, 70)])
def test_prefill_dense_params(oracle_mod, shape, T):
    """Head size 128: the one-grid form (chunk units and chains together);
    head size 32: the CUDA-core form."""
    B = 2
    d = I.decode_batch(seed=163, B=B, shape=shape)
    acts = I.activations(shape, B, T, torch.Generator().manual_seed(164))
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S, B, T)
    gdn.check_status()
    ref = _reference(oracle_mod, shape, d, acts, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])


def test_prefill_packed_params(oracle_mod):
    """Head size 128, three packed rows: the separate chunk and state kernels,
    the state kernel forming the outputs."""
    shape = I.Shape(nk=2, nv=4, dk=128, dv=128)
    real = [70, 130, 16]
    padded = [(n + 15) // 16 * 16 for n in real]
    cu = [0]
    for p in padded:
        cu.append(cu[-1] + p)
    total, B = cu[-1], len(real)
    d = I.decode_batch(seed=165, B=B, shape=shape)
    acts = I.activations(shape, 1, total, torch.Generator().manual_seed(166))
    mask = torch.zeros((1, total))
    for r in range(B):
        mask[0, cu[r]:cu[r] + real[r]] = 1.0
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S, B, total, mask=dev(mask),
                   cu=torch.tensor(cu, dtype=torch.int32, device="cuda"))
    gdn.check_status()
    out_h, S_h = out.cpu(), S.cpu()
    for r in range(B):
        a, b_ = cu[r], cu[r + 1]
        ra = {n: acts[n][:, a:b_] for n in ACTS}
        ref = _reference(oracle_mod, shape, d, ra, d["conv_state"][r:r + 1], d["state"][r:r + 1],
                         mask=mask[:, a:b_], real=real[r])
        assert_out(out_h[:, a:a + real[r]], ref["out"][:, :real[r]], f"row {r}")
        assert_state(S_h[r], ref["state"][0], f"row {r}")
