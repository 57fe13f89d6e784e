"""GPU parity of gdn_prefill_chunked against the fp64 oracle, through the C-ABI:
a long row continued in 512-token calls, packed varlen rows padded to chunk
buckets, short rows (conv tail shorter than the kernel), ragged tails."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from tests.gpu_cases import ACTS, WEIGHTS, assert_out, assert_state, dev, dims, inputs, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    build.build()
    gdn.load_library()


def _wd(d):
    return {n: dev(d[n]) for n in WEIGHTS}


def _prefill(shape, w, acts, conv, S, mask=None, cu=None, B=None, state_idx=None, n_slots=None):
    Bx, T = acts["q"].shape[0], acts["q"].shape[1]
    B = Bx if B is None else B
    out = torch.empty((Bx, T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    dm = dims(shape, B, T, n_slots or conv.shape[0])
    ws = gdn.workspace(dm, packed=cu is not None)  # exactly the size the layout needs
    gdn.prefill_chunked(dm, inputs(w, acts, mask=mask, cu=cu, state_idx=state_idx), conv, S, out, ws)
    return out


def test_long_row_in_512_token_calls(oracle_mod):
    """T=8192 continued from a saved state in 16 calls of 512 tokens, against
    one uninterrupted oracle pass."""
    d = I.prefill_long(seed=2)
    s = d["shape"]
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    outs = []
    for c in range(16):
        sl = slice(512 * c, 512 * (c + 1))
        outs.append(_prefill(s, w, {n: dev(d[n][:, sl].contiguous()) for n in ACTS}, conv, S))
    gdn.check_status()
    out = torch.cat(outs, 1)
    ref = oracle_layer(oracle_mod, s, d, d, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


@pytest.mark.parametrize("T", [1, 2, 3, 5, 64, 100, 130])
def test_ragged_lengths_and_short_tails(oracle_mod, T):
    """Lengths below the conv width, exactly one chunk, and ragged tails."""
    shape = I.TINY
    d = I.decode_batch(seed=30 + T, B=3, shape=shape)
    g = torch.Generator().manual_seed(T)
    acts = I.activations(shape, 3, T, g)
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, shape, d, acts, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


@pytest.mark.parametrize("shape", [I.Shape(nk=4, nv=8, dk=64, dv=64), I.Shape(nk=2, nv=4, dk=128, dv=128)])
def test_head_sizes_with_padding(oracle_mod, shape):
    d = I.decode_batch(seed=40, B=3, shape=shape)
    T = 150
    acts = I.activations(shape, 3, T, torch.Generator().manual_seed(41))
    mask = torch.zeros((3, T))
    for r, Lr in enumerate((150, 77, 0)):
        mask[r, :Lr] = 1
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S, mask=dev(mask))
    gdn.check_status()
    ref = oracle_layer(oracle_mod, shape, d, acts, d["conv_state"], d["state"], mask=mask)
    for r, Lr in enumerate((150, 77, 0)):
        assert_out(out[r, :Lr], ref["out"][r, :Lr])
        assert torch.count_nonzero(out[r, Lr:]) == 0
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))
    # the row with no real token is untouched bit for bit
    assert torch.equal(S[2].cpu(), d["state"][2]) and torch.equal(conv[2].cpu(), d["conv_state"][2])


@pytest.mark.parametrize("layer", range(24))
def test_varlen_layer_stack(oracle_mod, layer):
    """The packed varlen workload as the benchmark runs it, layer by layer: 32
    rows, lengths U{16..2048} padded to chunk buckets (mask 0 on the padding),
    each from its own state, with the layer's own weights and inputs drawn on
    the device by the same seeded generator. Every row of every one of the 24
    layers against the oracle: outputs at real tokens, zeros at padding, the
    final state and the conv tail (bit for bit)."""
    from concurrent.futures import ThreadPoolExecutor
    d = I.varlen_layer(layer, device="cuda")
    s = d["shape"]
    cu = d["cu_seqlens"]
    acts = {n: d[n] for n in ACTS}
    conv, S = d["conv_state"].clone(), d["state"].clone()
    out = _prefill(s, {n: d[n] for n in WEIGHTS}, acts, conv, S, mask=d["mask"][0], cu=cu.to("cuda"), B=32)
    gdn.check_status()
    h = {n: d[n].cpu() for n in ACTS + WEIGHTS}
    conv0, S0, mask = d["conv_state"].cpu(), d["state"].cpu(), d["mask"].cpu()
    out_h, S_h, conv_h = out.cpu(), S.cpu(), conv.cpu()
    del d, acts, out, S, conv
    real = I.varlen_lengths()[0]

    def row(r):
        a, b_ = int(cu[r]), int(cu[r + 1])
        ra = {n: h[n][:, a:b_] for n in ACTS}
        return r, oracle_layer(oracle_mod, s, h, ra, conv0[r:r + 1], S0[r:r + 1], mask=mask[:, a:b_])

    order = sorted(range(32), key=lambda r: -real[r])  # longest rows first
    with ThreadPoolExecutor(max_workers=4) as ex:
        for r, ref in ex.map(row, order):
            a, b_ = int(cu[r]), int(cu[r + 1])
            Lr = real[r]
            assert_out(out_h[:, a:a + Lr], ref["out"][:, :Lr], f"layer {layer} row {r}")
            assert torch.count_nonzero(out_h[:, a + Lr:b_]) == 0
            assert_state(S_h[r], ref["state"][0], f"layer {layer} row {r}")
            assert torch.equal(conv_h[r].double(), torch.from_numpy(ref["conv_state"][0]))


def test_split_call_equals_whole_call(oracle_mod):
    shape = I.TINY
    d = I.decode_batch(seed=50, B=2, shape=shape)
    acts = {n: dev(a) for n, a in I.activations(shape, 2, 192, torch.Generator().manual_seed(51)).items()}
    w = _wd(d)
    c1, S1 = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    whole = _prefill(shape, w, acts, c1, S1)
    c2, S2 = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    parts = [_prefill(shape, w, {n: a[:, sl].contiguous() for n, a in acts.items()}, c2, S2)
             for sl in (slice(0, 64), slice(64, 101), slice(101, 192))]
    gdn.check_status()
    assert torch.equal(c1, c2)
    assert_state(S2, S1.cpu().double().numpy())
    assert_out(torch.cat(parts, 1), whole.cpu().double().numpy())


@pytest.mark.parametrize("T", [1, 3, 64, 130])
def test_tensor_core_path_short_and_ragged(oracle_mod, T):
    """Head size 128 (the tcgen05 chunked path): rows shorter than the conv
    width, exactly one chunk, and a ragged last chunk."""
    shape = I.Shape(nk=2, nv=4, dk=128, dv=128)
    d = I.decode_batch(seed=70 + T, B=3, shape=shape)
    acts = I.activations(shape, 3, T, torch.Generator().manual_seed(71 + T))
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, shape, d, acts, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


@pytest.mark.parametrize("nk,nv", [(2, 2), (1, 4)])
def test_tensor_core_path_gqa_groups(oracle_mod, nk, nv):
    """Head size 128 with one value head per key head (G=1) and four (G=4):
    the key-head mapping, the per-key-head K^T image and the conv-tail update
    of the shared q|k channels."""
    shape = I.Shape(nk=nk, nv=nv, dk=128, dv=128)
    d = I.decode_batch(seed=80 + nv, B=2, shape=shape)
    T = 100
    acts = I.activations(shape, 2, T, torch.Generator().manual_seed(81 + nv))
    mask = torch.ones((2, T))
    mask[1, 61:] = 0
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S, mask=dev(mask))
    gdn.check_status()
    ref = oracle_layer(oracle_mod, shape, d, acts, d["conv_state"], d["state"], mask=mask)
    assert_out(out[0], ref["out"][0])
    assert_out(out[1, :61], ref["out"][1, :61])
    assert torch.count_nonzero(out[1, 61:].float()) == 0
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


def test_tensor_core_path_rejected_row(oracle_mod):
    """Head size 128, three rows in one call (the chunk and state passes then
    share one grid): a row whose mask is not ones then zeros is reported
    (GDN_ERR_MASK) and skipped -- its state, conv tail and outputs are not
    written -- while the other rows match the oracle."""
    shape = I.Shape(nk=2, nv=4, dk=128, dv=128)
    d = I.decode_batch(seed=90, B=3, shape=shape)
    T = 130
    acts = I.activations(shape, 3, T, torch.Generator().manual_seed(91))
    mask = torch.ones((3, T))
    mask[1, 40] = 0  # a hole: not a prefix of ones
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = torch.full((3, T, shape.nv, shape.dv), 7.0, dtype=torch.bfloat16, device="cuda")
    dm = dims(shape, 3, T, 3)
    ws = gdn.workspace(dm)
    dacts = {n: dev(a) for n, a in acts.items()}
    gdn.prefill_chunked(dm, inputs(w, dacts, mask=dev(mask)), conv, S, out, ws)
    with pytest.raises(gdn.GdnError) as e:
        gdn.check_status()
    assert e.value.name == "GDN_ERR_MASK"
    assert torch.equal(S[1].cpu(), d["state"][1]) and torch.equal(conv[1].cpu(), d["conv_state"][1])
    assert bool(torch.all(out[1].float() == 7.0))
    for r in (0, 2):
        ra = {n: a[r:r + 1] for n, a in acts.items()}
        ref = oracle_layer(oracle_mod, shape, d, ra, d["conv_state"][r:r + 1], d["state"][r:r + 1])
        assert_out(out[r:r + 1], ref["out"], f"row {r}")
        assert_state(S[r], ref["state"][0], f"row {r}")
        assert torch.equal(conv[r].cpu().double(), torch.from_numpy(ref["conv_state"][0]))


def test_many_chains_rejected_and_padded_rows(oracle_mod):
    """Head size 128, 40 rows x 4 value heads: 160 chains, so the chunk and
    state passes run as separate kernels and the state pass forms the outputs
    itself. A row whose mask is not ones then zeros is reported (GDN_ERR_MASK)
    and skipped -- its state, conv tail and outputs are not written; a padded
    row gets zeros after its real length; every other row matches the oracle."""
    shape = I.Shape(nk=2, nv=4, dk=128, dv=128)
    B, T = 40, 70
    d = I.decode_batch(seed=95, B=B, shape=shape)
    acts = I.activations(shape, B, T, torch.Generator().manual_seed(96))
    mask = torch.ones((B, T))
    mask[7, 20] = 0   # a hole: not a prefix of ones
    mask[11, 33:] = 0  # padding after 33 real tokens
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = torch.full((B, T, shape.nv, shape.dv), 7.0, dtype=torch.bfloat16, device="cuda")
    dm = dims(shape, B, T, B)
    ws = gdn.workspace(dm)
    gdn.prefill_chunked(dm, inputs(w, {n: dev(a) for n, a in acts.items()}, mask=dev(mask)), conv, S, out, ws)
    with pytest.raises(gdn.GdnError) as e:
        gdn.check_status()
    assert e.value.name == "GDN_ERR_MASK"
    assert torch.equal(S[7].cpu(), d["state"][7]) and torch.equal(conv[7].cpu(), d["conv_state"][7])
    assert bool(torch.all(out[7].float() == 7.0))
    keep = [r for r in range(B) if r != 7]
    ra = {n: a[keep] for n, a in acts.items()}
    dd = dict(d)
    ref = oracle_layer(oracle_mod, shape, dd, ra, d["conv_state"][keep], d["state"][keep], mask=mask[keep])
    o = out[keep]
    pad = keep.index(11)
    assert torch.count_nonzero(o[pad, 33:].float()) == 0
    o_real = torch.cat([o[:pad], o[pad + 1:]])
    ref_real = np.concatenate([ref["out"][:pad], ref["out"][pad + 1:]])
    assert_out(o_real, ref_real)
    assert_out(o[pad, :33], ref["out"][pad, :33])
    assert_state(S[keep], ref["state"])
    assert torch.equal(conv[keep].cpu().double(), torch.from_numpy(ref["conv_state"]))


def test_packed_rows_beyond_one_warp_of_offsets(oracle_mod):
    """Head size 128, 45 packed rows: the slot -> row lookup reads the row
    offsets 32 at a time, so rows 32-44 sit in a second window. Real lengths
    from 0 to 200 tokens (a row of padding only among them), each padded to a
    multiple of 16 with mask zeros, each row from its own state: outputs at
    real tokens, zeros at padding, final states and conv tails (bit for bit)
    against the oracle, row by row."""
    shape = I.Shape(nk=2, nv=4, dk=128, dv=128)
    B = 45
    real = [(37 * r + 11) % 201 for r in range(B)]
    real[20] = 0                  # padding only: the row stays as it was
    real[3], real[40] = 64, 129   # a whole chunk, and one token past two
    padded = [max(16, (n + 15) // 16 * 16) for n in real]
    cu = [0]
    for p in padded:
        cu.append(cu[-1] + p)
    total = cu[-1]
    d = I.decode_batch(seed=97, B=B, shape=shape)
    acts = I.activations(shape, 1, total, torch.Generator().manual_seed(98))
    mask = torch.zeros((1, total))
    for r in range(B):
        mask[0, cu[r]:cu[r] + real[r]] = 1.0
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S, mask=dev(mask), cu=cu_d, B=B)
    gdn.check_status()
    out_h, S_h, conv_h = out.cpu(), S.cpu(), conv.cpu()
    for r in range(B):
        a, b_ = cu[r], cu[r + 1]
        Lr = real[r]
        assert torch.count_nonzero(out_h[:, a + Lr:b_]) == 0, f"row {r}"
        if Lr == 0:
            assert torch.equal(S_h[r], d["state"][r]) and torch.equal(conv_h[r], d["conv_state"][r])
            continue
        ra = {n: acts[n][:, a:b_] for n in ACTS}
        ref = oracle_layer(oracle_mod, shape, d, ra, d["conv_state"][r:r + 1], d["state"][r:r + 1],
                           mask=mask[:, a:b_])
        assert_out(out_h[:, a:a + Lr], ref["out"][:, :Lr], f"row {r}")
        assert_state(S_h[r], ref["state"][0], f"row {r}")
        assert torch.equal(conv_h[r].double(), torch.from_numpy(ref["conv_state"][0]))


@pytest.mark.parametrize("B", [19, 20])
def test_chain_grid_boundary(oracle_mod, B):
    """Head size 128, 4 value heads, two chunks per row. 19 rows make 76
    chains on a grid of 152 chunk units: the few-chain grid at its limit, half
    of its CTAs running chains (each first runs its own chain's first chunk)
    and the other half the second chunks. 20 rows (80 chains) take the
    separate chunk and state kernels. Both against the oracle."""
    shape = I.Shape(nk=2, nv=4, dk=128, dv=128)
    T = 128
    d = I.decode_batch(seed=99 + B, B=B, shape=shape)
    acts = I.activations(shape, B, T, torch.Generator().manual_seed(100 + B))
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, shape, d, acts, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


@pytest.mark.parametrize("shape,packed", [(I.Shape(nk=2, nv=4, dk=128, dv=128), False),
                                          (I.Shape(nk=2, nv=4, dk=128, dv=128), True), (I.TINY, False)])
def test_state_pool_slots(oracle_mod, shape, packed):
    """Rows continue from pool slots chosen by state_idx (3 rows over 7 slots,
    out of order): every path reads and writes its row's slot -- the one-grid
    tensor-core form (dense rows), the separate-kernel form (packed rows) and
    the CUDA-core form (head size 32) -- and the 4 unused slots stay as they
    were, bit for bit."""
    B, n_slots = 3, 7
    idx = torch.tensor([5, 0, 3], dtype=torch.int32)
    g = torch.Generator().manual_seed(170)
    pool = I.states(shape, n_slots, g)
    d = I.decode_batch(seed=171, B=B, shape=shape)
    w = _wd(d)
    conv, S = dev(pool["conv_state"]).clone(), dev(pool["state"]).clone()
    if packed:
        real = [70, 16, 129]
        cu = [0]
        for n in real:
            cu.append(cu[-1] + (n + 15) // 16 * 16)
        acts = I.activations(shape, 1, cu[-1], g)
        mask = torch.zeros((1, cu[-1]))
        for r in range(B):
            mask[0, cu[r]:cu[r] + real[r]] = 1.0
        out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S, mask=dev(mask),
                       cu=torch.tensor(cu, dtype=torch.int32, device="cuda"), B=B, state_idx=dev(idx),
                       n_slots=n_slots)
    else:
        T = 100
        acts = I.activations(shape, B, T, g)
        out = _prefill(shape, w, {n: dev(a) for n, a in acts.items()}, conv, S, state_idx=dev(idx), n_slots=n_slots)
    gdn.check_status()
    out_h, S_h, conv_h = out.cpu(), S.cpu(), conv.cpu()
    for r in range(B):
        sl = int(idx[r])
        c0, s0 = pool["conv_state"][sl:sl + 1], pool["state"][sl:sl + 1]
        if packed:
            a, b_ = cu[r], cu[r + 1]
            ref = oracle_layer(oracle_mod, shape, d, {n: acts[n][:, a:b_] for n in ACTS}, c0, s0, mask=mask[:, a:b_])
            assert_out(out_h[:, a:a + real[r]], ref["out"][:, :real[r]], f"row {r}")
        else:
            ref = oracle_layer(oracle_mod, shape, d, {n: acts[n][r:r + 1] for n in ACTS}, c0, s0)
            assert_out(out_h[r:r + 1], ref["out"], f"row {r}")
        assert_state(S_h[sl], ref["state"][0], f"row {r} (slot {sl})")
        assert torch.equal(conv_h[sl].double(), torch.from_numpy(ref["conv_state"][0])), f"row {r} conv tail"
    for sl in sorted(set(range(n_slots)) - set(idx.tolist())):
        assert torch.equal(S_h[sl], pool["state"][sl]) and torch.equal(conv_h[sl], pool["conv_state"][sl]), sl
