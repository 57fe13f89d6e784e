"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
hand-worked examples, textbook/library routines, closed forms and invariants of
the Gated DeltaNet layer (statecache.py, squad-0.8b: CacheQwen35._gdn; generate.py,
sparkle mlx_streaming/mtp: per-token verify checkpoints)."""
import json
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gated_deltanet_recurrence_delta_gb300 import inputs as I
from tests.wy_chunked import chunked_recurrence

GOLDEN = Path(__file__).parent / "golden"


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


# ------------------------------------------------------------------ golden

def test_delta_rule_hand_example(oracle_mod):
    d = json.loads((GOLDEN / "delta_rule_2x2_hand.json").read_text())
    o, S, ck = oracle_mod.recurrence(np.array(d["q"]), np.array(d["k"]), np.array(d["v"]),
                                     np.array(d["g"]), np.array(d["beta"]), np.array(d["S0"]),
                                     ckpt=True)
    tol = d["tolerance"]
    np.testing.assert_allclose(o, np.array(d["expected_o"]), atol=tol, rtol=0)
    np.testing.assert_allclose(ck, np.array(d["expected_ckpt"]), atol=tol, rtol=0)
    np.testing.assert_allclose(S, np.array(d["expected_ckpt"])[-1], atol=tol, rtol=0)


def test_conv_tail_hand_example(oracle_mod):
    d = json.loads((GOLDEN / "conv_tail_hand.json").read_text())
    x = np.array(d["x"])[:, None]
    w = np.array(d["w"])[None, :]
    tail = np.array(d["tail"])[:, None]
    for Lr, expect_tail in d["expected_tail"].items():
        y, new_tail, _ = oracle_mod.conv(x, w, tail, Lr=int(Lr))
        pre = np.array(d["expected_preact"])
        np.testing.assert_allclose(y[:, 0], pre / (1 + np.exp(-pre)), rtol=1e-15)
        np.testing.assert_array_equal(new_tail[:, 0], np.array(expect_tail))


# ------------------------------------------------------- library routines

def test_conv_matches_torch_conv1d(oracle_mod):
    r = _rng(1)
    T, C, K = 37, 24, 4
    x = r.standard_normal((T, C))
    w = r.standard_normal((C, K)) * 0.25
    tail = r.standard_normal((K - 1, C))
    y, new_tail, ck = oracle_mod.conv(x, w, tail, ckpt=True)
    xin = torch.from_numpy(np.concatenate([tail, x], 0).T[None])       # [1, C, K-1+T]
    ref = F.conv1d(xin, torch.from_numpy(w)[:, None, :], groups=C)     # [1, C, T]
    ref = F.silu(ref)[0].T.numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(new_tail, x[-(K - 1):])
    # the tail checkpoint after token t is the last K-1 inputs up to t
    xin_np = np.concatenate([tail, x], 0)
    for t in range(T):
        np.testing.assert_array_equal(ck[t], xin_np[t + 1:t + K])


def test_conv_current_token_tap(oracle_mod):
    """w = e_{K-1}: only the current token contributes, so y = silu(x) exactly."""
    r = _rng(2)
    x = r.standard_normal((9, 5))
    w = np.zeros((5, 4)); w[:, 3] = 1.0
    y, _, _ = oracle_mod.conv(x, w, r.standard_normal((3, 5)))
    np.testing.assert_allclose(y, x / (1 + np.exp(-x)), rtol=1e-15, atol=0)


@pytest.mark.parametrize("Lr", [0, 1, 2, 3, 7])
def test_conv_tail_short_chunks(oracle_mod, Lr):
    """The tail keeps old rows when fewer than K-1 real inputs arrive."""
    r = _rng(3)
    x = r.standard_normal((7, 6)); tail = r.standard_normal((3, 6))
    _, new_tail, _ = oracle_mod.conv(x, np.ones((6, 4)), tail, Lr=Lr)
    xin = np.concatenate([tail, x], 0)
    np.testing.assert_array_equal(new_tail, xin[Lr:Lr + 3])


def test_gates_match_torch(oracle_mod):
    r = _rng(4)
    T, nv = 50, 6
    a = r.standard_normal((T, nv)) * 8
    b = r.standard_normal((T, nv)) * 4
    A_log = np.log(r.uniform(1, 16, nv)); dt_bias = r.uniform(-1, 1, nv)
    mask = np.ones(T); mask[40:] = 0
    g, beta = oracle_mod.gates(a, b, A_log, dt_bias, mask)
    at, bt = torch.from_numpy(a), torch.from_numpy(b)
    # torch.softplus returns x above its threshold; use a threshold no input reaches
    g_ref = -torch.exp(torch.from_numpy(A_log)) * F.softplus(at + torch.from_numpy(dt_bias), threshold=1e4)
    beta_ref = torch.sigmoid(bt)
    m = torch.from_numpy(mask)[:, None]
    np.testing.assert_allclose(g, (g_ref * m).numpy(), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(beta, (beta_ref * m).numpy(), rtol=1e-14, atol=0)
    assert np.all(g[40:] == 0) and np.all(beta[40:] == 0)
    assert np.all(g[:40] < 0) and np.all((beta[:40] > 0) & (beta[:40] < 1))


def test_l2norm_matches_torch_normalize(oracle_mod):
    r = _rng(5)
    x = r.standard_normal(128) * 3
    out = oracle_mod.l2norm(x, eps=0.0, scale=1.0)
    np.testing.assert_allclose(out, F.normalize(torch.from_numpy(x), dim=0).numpy(), rtol=1e-15, atol=1e-16)
    # with eps the squared norm is ss / (ss + eps), and scale multiplies after
    eps = 1e-3
    out = oracle_mod.l2norm(x, eps=eps, scale=0.5)
    ss = float(np.sum(x * x))
    np.testing.assert_allclose(np.sum(out * out), 0.25 * ss / (ss + eps), rtol=1e-14)


def test_gated_rmsnorm_matches_torch(oracle_mod):
    r = _rng(6)
    o = r.standard_normal(128); z = r.standard_normal(128); w = 1 + 0.1 * r.standard_normal(128)
    out = oracle_mod.gated_rmsnorm(o, z, w, eps=1e-6)
    ref = F.rms_norm(torch.from_numpy(o)[None], (128,), torch.from_numpy(w), eps=1e-6)[0] * F.silu(torch.from_numpy(z))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------- recurrence

def test_write_invariant(oracle_mod):
    """g = 0, beta = 1, unit key: after the write the state maps k to v."""
    r = _rng(7)
    dk, dv = 16, 12
    S0 = r.standard_normal((dk, dv))
    k = _unit(r.standard_normal((1, dk)))
    v = r.standard_normal((1, dv))
    q = r.standard_normal((1, dk))
    o, S, _ = oracle_mod.recurrence(q, k, v, np.zeros(1), np.ones(1), S0)
    np.testing.assert_allclose(S.T @ k[0], v[0], atol=1e-12)
    np.testing.assert_allclose(o[0], S.T @ q[0], atol=1e-12)


def test_beta_zero_closed_form(oracle_mod):
    """beta = 0: pure decay, S_T = exp(sum g) S_0, o_t = exp(G_t) S_0^T q_t."""
    r = _rng(8)
    T, dk, dv = 20, 8, 8
    S0 = r.standard_normal((dk, dv))
    q = r.standard_normal((T, dk)); k = _unit(r.standard_normal((T, dk))); v = r.standard_normal((T, dv))
    g = -r.uniform(0, 0.5, T)
    o, S, _ = oracle_mod.recurrence(q, k, v, g, np.zeros(T), S0)
    G = np.cumsum(g)
    np.testing.assert_allclose(S, np.exp(G[-1]) * S0, rtol=1e-13)
    np.testing.assert_allclose(o, np.exp(G)[:, None] * (q @ S0), rtol=1e-12, atol=1e-14)


def test_scalar_geometric_closed_form(oracle_mod):
    """dk = dv = 1 with constant gates: S_t = a S_{t-1} + c, a = e^g (1 - beta k^2),
    c = beta k v, whose closed form is a^T S_0 + c (1 - a^T) / (1 - a)."""
    T = 30
    g, beta, kk, vv, S0 = -0.2, 0.3, -1.0, 2.5, 0.7
    o, S, ck = oracle_mod.recurrence(np.ones((T, 1)), np.full((T, 1), kk), np.full((T, 1), vv),
                                     np.full(T, g), np.full(T, beta), np.array([[S0]]), ckpt=True)
    a = np.exp(g) * (1 - beta * kk * kk)
    c = beta * kk * vv
    t = np.arange(1, T + 1)
    closed = a ** t * S0 + c * (1 - a ** t) / (1 - a)
    np.testing.assert_allclose(ck[:, 0, 0], closed, rtol=1e-13)
    np.testing.assert_allclose(o[:, 0], closed, rtol=1e-13)


def test_matrix_form_orientation(oracle_mod):
    """The rule as a matrix product on S [dv, dk]:
    S_t = e^g S_{t-1} (I - beta k k^T) + beta v k^T, o = S q; the oracle keeps the
    transpose.  A transposed operand or a swapped k/q fails this."""
    r = _rng(9)
    T, dk, dv = 6, 5, 3
    S = r.standard_normal((dv, dk))
    q = r.standard_normal((T, dk)); k = _unit(r.standard_normal((T, dk))); v = r.standard_normal((T, dv))
    g = -r.uniform(0, 1, T); beta = r.uniform(0, 1, T)
    o, St, _ = oracle_mod.recurrence(q, k, v, g, beta, S.T.copy())
    for t in range(T):
        S = np.exp(g[t]) * S @ (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) + beta[t] * np.outer(v[t], k[t])
        np.testing.assert_allclose(o[t], S @ q[t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(St, S.T, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
@pytest.mark.parametrize("gscale", ["config", "slow"])
def test_chunked_wy_equals_token_recurrence(oracle_mod, chunk, gscale):
    """Brute force: the chunked WY form equals the token recurrence, including a
    partial last chunk (T = 130) and padded tokens (g = beta = 0)."""
    r = _rng(10 + chunk)
    T, dk, dv = 130, 16, 12
    q = _unit(r.standard_normal((T, dk))) * dk ** -0.5
    k = _unit(r.standard_normal((T, dk)))
    v = r.standard_normal((T, dv))
    if gscale == "config":
        g = -np.exp(np.log(r.uniform(1, 16, T))) * np.log1p(np.exp(r.standard_normal(T) + r.uniform(-1, 1, T)))
    else:
        g = -r.uniform(0, 0.05, T)
    beta = 1 / (1 + np.exp(-r.standard_normal(T)))
    g[120:] = 0; beta[120:] = 0
    S0 = r.standard_normal((dk, dv)) * 0.1
    o_tok, S_tok, _ = oracle_mod.recurrence(q, k, v, g, beta, S0)
    o_wy, S_wy = chunked_recurrence(q, k, v, g, beta, S0, chunk)
    scale = max(1.0, np.abs(o_tok).max())
    np.testing.assert_allclose(o_wy, o_tok, atol=1e-10 * scale, rtol=0)
    np.testing.assert_allclose(S_wy, S_tok, atol=1e-10 * max(1.0, np.abs(S_tok).max()), rtol=0)


# --------------------------------------------------------------- layer

def _tiny(T=64, seed=0):
    d = I.tiny_layer(seed)
    s = d["shape"]
    act = d["prefill"]
    kw = dict(A_log=d["A_log"], dt_bias=d["dt_bias"], conv_w=d["conv_w"], norm_w=d["norm_w"],
              nk=s.nk, nv=s.nv, dk=s.dk, dv=s.dv)
    acts = {n: t[:, :T] for n, t in act.items()}
    # a non-zero tail makes the continuation checks stronger
    conv = torch.randn(d["conv_state"].shape, generator=torch.Generator().manual_seed(seed + 99)).to(torch.bfloat16)
    return s, acts, kw, conv, d["state"]


def test_layer_mask_zero_leaves_state(oracle_mod):
    s, acts, kw, conv, S0 = _tiny(16)
    res = oracle_mod.layer(**acts, **kw, conv_state=conv, state=S0, mask=np.zeros((1, 16)))
    np.testing.assert_array_equal(res["state"], S0.double().numpy())
    np.testing.assert_array_equal(res["conv_state"], conv.double().numpy())


def test_layer_padding_stops_at_real_end(oracle_mod):
    """A padded row (mask = 1^Lr 0^pad) ends in the same state and conv tail as
    the unpadded row of Lr tokens, and agrees on the real outputs."""
    s, acts, kw, conv, S0 = _tiny(24)
    for Lr in (0, 1, 2, 5, 23):
        mask = np.zeros((1, 24)); mask[0, :Lr] = 1
        padded = oracle_mod.layer(**acts, **kw, conv_state=conv, state=S0, mask=mask)
        real = oracle_mod.layer(**{n: t[:, :Lr] for n, t in acts.items()}, **kw, conv_state=conv, state=S0)
        np.testing.assert_array_equal(padded["state"], real["state"])
        np.testing.assert_array_equal(padded["conv_state"], real["conv_state"])
        np.testing.assert_array_equal(padded["out"][:, :Lr], real["out"])


def test_layer_rejects_non_prefix_mask(oracle_mod):
    s, acts, kw, conv, S0 = _tiny(8)
    mask = np.ones((1, 8)); mask[0, 3] = 0
    with pytest.raises(ValueError):
        oracle_mod.layer(**acts, **kw, conv_state=conv, state=S0, mask=mask)


@pytest.mark.parametrize("split", [1, 3, 16, 40])
def test_layer_split_continuation_bitwise(oracle_mod, split):
    """Splitting a sequence anywhere and continuing from the saved conv tail and
    state gives the whole-sequence result bit for bit."""
    s, acts, kw, conv, S0 = _tiny(64)
    whole = oracle_mod.layer(**acts, **kw, conv_state=conv, state=S0)
    first = oracle_mod.layer(**{n: t[:, :split] for n, t in acts.items()}, **kw, conv_state=conv, state=S0)
    second = oracle_mod.layer(**{n: t[:, split:] for n, t in acts.items()}, **kw,
                              conv_state=first["conv_state"], state=first["state"])
    np.testing.assert_array_equal(np.concatenate([first["out"], second["out"]], 1), whole["out"])
    np.testing.assert_array_equal(second["state"], whole["state"])
    np.testing.assert_array_equal(second["conv_state"], whole["conv_state"])


def test_layer_checkpoints_equal_prefix_runs(oracle_mod):
    """Verify checkpoint j equals the state after j+1 tokens (bitwise), and the
    conv checkpoint equals that run's conv tail."""
    s, acts, kw, conv, S0 = _tiny(8)
    full = oracle_mod.layer(**acts, **kw, conv_state=conv, state=S0, checkpoints=True)
    for j in range(8):
        part = oracle_mod.layer(**{n: t[:, :j + 1] for n, t in acts.items()}, **kw, conv_state=conv, state=S0)
        np.testing.assert_array_equal(full["ckpt_state"][0, j], part["state"][0])
        np.testing.assert_array_equal(full["ckpt_conv"][0, j], part["conv_state"][0])


def test_layer_gqa_equals_expanded_heads(oracle_mod):
    """GQA (nk=2, nv=4) equals the layer with nk = nv whose q/k channels, conv
    weights and conv tail are the key heads repeated per value head
    (repeat_interleave by nv/nk)."""
    s, acts, kw, conv, S0 = _tiny(12)
    G = s.nv // s.nk
    gqa = oracle_mod.layer(**acts, **kw, conv_state=conv, state=S0)

    def rep(x, axis):  # [.., nk*dk] -> [.., nv*dk] with each key head repeated G times
        sh = list(x.shape)
        y = x.reshape(sh[:axis] + [s.nk, s.dk] + sh[axis + 1:])
        y = np.repeat(y, G, axis=axis)
        return y.reshape(sh[:axis] + [s.nv * s.dk] + sh[axis + 1:])

    qn, kn, vn = (acts[n].double().numpy() for n in ("q", "k", "v"))
    w = kw["conv_w"].double().numpy()
    kd = s.kd
    w_exp = np.concatenate([rep(w[:kd].T, 1).T, rep(w[kd:2 * kd].T, 1).T, w[2 * kd:]], 0)
    c = conv.double().numpy()
    c_exp = np.concatenate([rep(c[:, :, :kd], 2), rep(c[:, :, kd:2 * kd], 2), c[:, :, 2 * kd:]], 2)
    kw2 = dict(kw); kw2.update(nk=s.nv, conv_w=w_exp)
    exp = oracle_mod.layer(q=rep(qn, 2), k=rep(kn, 2), v=vn, z=acts["z"], a=acts["a"], b=acts["b"],
                           **{k_: v_ for k_, v_ in kw2.items()}, conv_state=c_exp, state=S0)
    np.testing.assert_array_equal(gqa["out"], exp["out"])
    np.testing.assert_array_equal(gqa["state"], exp["state"])


def test_layer_rows_independent(oracle_mod):
    """Row b of a batched call equals the single-row call on that row."""
    d = I.decode_batch(seed=5, B=3, shape=I.TINY)
    s = d["shape"]
    kw = dict(A_log=d["A_log"], dt_bias=d["dt_bias"], conv_w=d["conv_w"], norm_w=d["norm_w"],
              nk=s.nk, nv=s.nv, dk=s.dk, dv=s.dv)
    acts = {n: d[n] for n in ("q", "k", "v", "z", "a", "b")}
    full = oracle_mod.layer(**acts, **kw, conv_state=d["conv_state"], state=d["state"])
    for b in range(3):
        one = oracle_mod.layer(**{n: t[b:b + 1] for n, t in acts.items()}, **kw,
                               conv_state=d["conv_state"][b:b + 1], state=d["state"][b:b + 1])
        np.testing.assert_array_equal(full["out"][b], one["out"][0])
        np.testing.assert_array_equal(full["state"][b], one["state"][0])
