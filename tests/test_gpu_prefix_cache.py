"""The prefix state cache on the GPU (statecache.py, squad-0.8b, StateCache),
through the C-ABI:

  - gdn_prefill_chunked_ckpt writes, from inside the prefill, the state and
    conv tail of a row after its first p tokens (p a chunk end or the real end;
    p < 3 takes rows of the saved tail) into the requested slots: each equals
    the oracle run over those p tokens; the call's own outputs, states and
    tails are those of gdn_prefill_chunked; bad triples are recorded
    (GDN_ERR_INDEX) and skipped. Head size 128 with dense rows (chunk and state
    passes in one grid) and packed rows (separate kernels), and head size 32.
  - PrefixStateCache over a two-layer stack: a cold row, a row sharing part of
    its prefix (restored from the deepest shared checkpoint by one
    gdn_state_copy launch, then continued), and the first row again (a hit):
    every output computed and every final state equal the oracle's
    uninterrupted pass over the whole row from a zero state."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from gated_deltanet_recurrence_delta_gb300.prefix_cache import PrefixStateCache
from gated_deltanet_recurrence_delta_gb300.stack import LayerStack
from tests.gpu_cases import ACTS, WEIGHTS, assert_out, assert_state, dev, dims, inputs, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    build.build()
    gdn.load_library()


@pytest.mark.parametrize("shape,packed", [(I.Shape(nk=2, nv=4, dk=128, dv=128), False),
                                          (I.Shape(nk=2, nv=4, dk=128, dv=128), True), (I.TINY, False)])
def test_prefill_checkpoints(oracle_mod, shape, packed):
    B, T = 3, 200
    lens = (200, 130, 2)
    d = I.decode_batch(seed=150 + int(packed), B=B, shape=shape)
    acts = I.activations(shape, B, T, torch.Generator().manual_seed(151))
    mask = torch.zeros((B, T))
    for r, L in enumerate(lens):
        mask[r, :L] = 1
    good = [(0, 64, 0), (0, 128, 1), (0, 192, 2), (0, 200, 3), (1, 64, 4), (1, 128, 5), (1, 130, 6), (2, 2, 7)]
    bad = [(0, 100, 8), (1, 192, 8), (5, 64, 8), (0, 64, 99)]  # not a chunk end, past Lr, no such row, no slot
    n_slots = 9
    trip = dev(torch.tensor(good + bad, dtype=torch.int32))
    ck_S = torch.zeros((n_slots, shape.nv, shape.dk, shape.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.zeros((n_slots, 3, shape.C), dtype=torch.bfloat16, device="cuda")
    w = {n: dev(d[n]) for n in WEIGHTS}
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    if packed:
        cu = dev(torch.tensor([0, T, 2 * T, 3 * T], dtype=torch.int32))
        pa = {n: dev(a.reshape(1, B * T, -1).contiguous()) for n, a in acts.items()}
        out = torch.zeros((1, B * T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
        dm = dims(shape, B, B * T, B)
        inp = inputs(w, pa, mask=dev(mask.reshape(-1)), cu=cu)
    else:
        out = torch.zeros((B, T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
        dm = dims(shape, B, T, B)
        inp = inputs(w, {n: dev(a) for n, a in acts.items()}, mask=dev(mask))
    gdn.prefill_chunked_ckpt(dm, inp, conv, S, out, gdn.workspace(dm, packed=packed), trip, ck_S, ck_c)
    with pytest.raises(gdn.GdnError) as e:
        gdn.check_status()
    assert e.value.name == "GDN_ERR_INDEX"
    out = out.reshape(B, T, shape.nv, shape.dv)
    # the call itself: as without checkpoints
    ref = oracle_layer(oracle_mod, shape, d, acts, d["conv_state"], d["state"], mask=mask)
    for r, L in enumerate(lens):
        assert_out(out[r, :L], ref["out"][r, :L], f"row {r}")
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))
    # each checkpoint: the oracle over the row's first p tokens
    for r, p, sl in good:
        rp = oracle_layer(oracle_mod, shape, d, {n: a[r:r + 1, :p] for n, a in acts.items()},
                          d["conv_state"][r:r + 1], d["state"][r:r + 1])
        assert_state(ck_S[sl], rp["state"][0], f"row {r} position {p}")
        assert torch.equal(ck_c[sl].cpu().double(), torch.from_numpy(rp["conv_state"][0])), f"row {r} position {p}"
    assert torch.count_nonzero(ck_S[8]) == 0 and torch.count_nonzero(ck_c[8]) == 0  # bad triples wrote nothing


@pytest.mark.parametrize("shape", [I.Shape(nk=2, nv=4, dk=128, dv=128), I.TINY])
def test_prefix_cache_rows(oracle_mod, shape):
    L, V = 2, 40
    g = torch.Generator().manual_seed(160)
    ws_cpu = [I.weights(shape, g) for _ in range(L)]
    # a token's inputs at each layer are a function of its id, so rows that
    # share tokens share inputs (and therefore states)
    table = [I.activations(shape, 1, V, g) for _ in range(L)]
    stack = LayerStack(shape, [{n: w[n].cuda() for n in WEIGHTS} for w in ws_cpu], n_slots=2)
    cache = PrefixStateCache(stack, mb=64, stride=128, tail=16)
    ws = gdn.workspace(dims(shape, 1, 512, 1))
    zero_c = torch.zeros((1, 3, shape.C), dtype=torch.bfloat16)
    zero_S = torch.zeros((1, shape.nv, shape.dk, shape.dv))

    def acts_of(ids):
        idx = torch.as_tensor(ids)
        return [{n: table[l][n][:, idx] for n in ACTS} for l in range(L)]

    def run(ids, state_len, slot, expect_c0):
        a = acts_of(ids)
        out = torch.zeros((L, 1, len(ids), shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
        c0 = cache.row(ids, state_len, [{n: t.cuda() for n, t in x.items()} for x in a], slot, out, ws)
        gdn.check_status()
        assert c0 == expect_c0
        for l in range(L):  # the uninterrupted pass over the whole row from zeros
            ref = oracle_layer(oracle_mod, shape, ws_cpu[l], a[l], zero_c, zero_S)
            assert_out(out[l][:, c0:], ref["out"][:, c0:], f"layer {l}")
            assert torch.count_nonzero(out[l][:, :c0]) == 0
            assert_state(stack.state_pool[l][slot], ref["state"][0], f"layer {l}")
            assert torch.equal(stack.conv_pool[l][slot].cpu().double(), torch.from_numpy(ref["conv_state"][0]))
        return a

    rng = np.random.default_rng(161)
    ids_a = rng.integers(0, V, 300)
    run(ids_a, 260, 0, 0)  # cold: checkpoints at 128, 192 (260 - 16, rounded down) and 256
    assert sorted(c.pos for c in cache.sched.ckpts.values()) == [128, 192, 256]
    ids_b = np.concatenate([ids_a[:200], rng.integers(0, V, 150)])
    ids_b[200] = (ids_a[200] + 1) % V  # shares exactly 200 tokens with row A
    a_b = run(ids_b, 330, 1, 192)  # restores A's checkpoint at 192, makes 256 and 320
    # row B's new checkpoints hold the oracle state after those tokens
    for c in cache.sched.ckpts.values():
        if c.group.ids.shape[0] == 320:
            for l in range(L):
                ref = oracle_layer(oracle_mod, shape, ws_cpu[l], {n: t[:, :c.pos] for n, t in a_b[l].items()},
                                   zero_c, zero_S)
                assert_state(cache.ckpt_state[l][c.slot], ref["state"][0], f"layer {l} position {c.pos}")
    run(ids_a, 260, 0, 256)  # row A again: a hit at its deepest checkpoint
    st = cache.sched.stats
    assert (st["cold"], st["partial"], st["hits"]) == (1, 1, 1)
