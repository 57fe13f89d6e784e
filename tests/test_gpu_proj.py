"""GPU parity of the layer's projections (gdn_in_proj, gdn_out_proj: tcgen05
GEMMs, the in-projection split into q, k, v, z, b, a in its epilogue) against
the oracle's fp64 products, through the C-ABI, and the projections around a
decode step.

Bar: each bf16 output within half a bf16 ulp of the exact product (its own
rounding) plus 1e-5 of the largest output (fp32 accumulation over K <= 4096
is far below that)."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from tests.gpu_cases import ACTS, WEIGHTS, assert_out, assert_state, bf16_half_ulp, dims, inputs, oracle_layer, record

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "z", "b", "a")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    build.build()
    gdn.load_library()


def _check(gpu, ref, what):
    g = gpu.detach().float().cpu().double().numpy().reshape(ref.shape)
    err = np.abs(g - ref) - bf16_half_ulp(ref)
    bar = 1e-5 * max(1.0, float(np.abs(ref).max()))
    worst = float(err.max()) if err.size else 0.0
    record("proj_beyond_half_ulp", worst)
    assert worst <= bar, f"{what}: {worst:.3e} beyond the bf16 rounding > {bar:.1e}"


def _weights(N, H, g):
    return (torch.randn((N, H), generator=g) * H ** -0.5).to(torch.bfloat16)


def _in_proj(shape, hidden, w_in):
    M = hidden.shape[0]
    outs = {"q": (M, shape.kd), "k": (M, shape.kd), "v": (M, shape.vd), "z": (M, shape.vd), "b": (M, shape.nv),
            "a": (M, shape.nv)}
    o = {n: torch.full(sh, 7.0, dtype=torch.bfloat16, device="cuda") for n, sh in outs.items()}
    gdn.in_proj(dims(shape, 1, 1, 1), hidden.cuda(), w_in.cuda(), o["q"], o["k"], o["v"], o["z"], o["a"], o["b"])
    return o


@pytest.mark.parametrize("M", [1, 3, 64, 65, 130, 300])
def test_in_proj_split_small(oracle_mod, M):
    """Tiny layer (2/4 heads, d=32: 392 features over 4 tiles, the last partial),
    H = 256; token counts from one to several tiles with ragged tails."""
    shape = I.TINY
    g = torch.Generator().manual_seed(200 + M)
    H = 256
    N = 2 * shape.kd + 2 * shape.vd + 2 * shape.nv
    hidden = torch.randn((M, H), generator=g).to(torch.bfloat16)
    w_in = _weights(N, H, g)
    o = _in_proj(shape, hidden, w_in)
    torch.cuda.synchronize()
    gdn.check_status()
    ref = oracle_mod.in_proj(hidden, w_in, shape.nk, shape.nv, shape.dk, shape.dv)
    for n in NAMES:
        _check(o[n], ref[n], n)


@pytest.mark.parametrize("M", [64, 100, 512])
def test_in_proj_qwen_layer(oracle_mod, M):
    """The Qwen3.5-9B-like layer: H = 4096, 12352 features (16/32 heads, d=128):
    one 64-token tile, one partial 128-token tile and two 256-token tiles, the
    last two in the grouped tile order (101 MB of weights)."""
    shape = I.QWEN35_9B
    g = torch.Generator().manual_seed(210 + M)
    H = 4096
    N = 2 * shape.kd + 2 * shape.vd + 2 * shape.nv
    hidden = torch.randn((M, H), generator=g).to(torch.bfloat16)
    w_in = _weights(N, H, g)
    o = _in_proj(shape, hidden, w_in)
    torch.cuda.synchronize()
    gdn.check_status()
    ref = oracle_mod.in_proj(hidden, w_in, shape.nk, shape.nv, shape.dk, shape.dv)
    for n in NAMES:
        _check(o[n], ref[n], n)


@pytest.mark.parametrize("M,H,V", [(1, 256, 128), (64, 4096, 4096), (200, 1000, 192)])
def test_out_proj(oracle_mod, M, H, V):
    g = torch.Generator().manual_seed(220 + M)
    o = torch.randn((M, V), generator=g).to(torch.bfloat16)
    w_out = _weights(H, V, g)
    y = torch.full((M, H), 7.0, dtype=torch.bfloat16, device="cuda")
    gdn.out_proj(o.cuda(), w_out.cuda(), y)
    torch.cuda.synchronize()
    gdn.check_status()
    _check(y, oracle_mod.out_proj(o, w_out), "y")


def test_projections_around_a_decode_step(oracle_mod):
    """hidden -> gdn_in_proj -> gdn_decode_step -> gdn_out_proj on the tiny
    layer, every stage against the oracle on the previous stage's GPU output."""
    shape = I.TINY
    B, H = 3, 256
    d = I.decode_batch(seed=230, B=B, shape=shape)
    g = torch.Generator().manual_seed(231)
    N = 2 * shape.kd + 2 * shape.vd + 2 * shape.nv
    hidden = torch.randn((B, H), generator=g).to(torch.bfloat16)
    w_in, w_out = _weights(N, H, g), _weights(H, shape.vd, g)
    o = _in_proj(shape, hidden, w_in)
    ref = oracle_mod.in_proj(hidden, w_in, shape.nk, shape.nv, shape.dk, shape.dv)
    for n in NAMES:
        _check(o[n], ref[n], n)
    acts = {n: o[n].view(B, 1, -1) for n in ACTS}
    w = {n: d[n].cuda() for n in WEIGHTS}
    conv, S = d["conv_state"].cuda().clone(), d["state"].cuda().clone()
    out = torch.empty((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    gdn.decode_step(dims(shape, B, 1, B), inputs(w, acts), conv, S, out)
    y = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    gdn.out_proj(out.view(B, shape.vd), w_out.cuda(), y)
    torch.cuda.synchronize()
    gdn.check_status()
    rl = oracle_layer(oracle_mod, shape, d, {n: t.cpu() for n, t in acts.items()}, d["conv_state"], d["state"])
    assert_out(out, rl["out"])
    assert_state(S, rl["state"])
    _check(y, oracle_mod.out_proj(out.view(B, shape.vd).cpu(), w_out), "y")
