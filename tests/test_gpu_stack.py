"""A stack of layers on per-layer state pools, stepped eagerly and from captured
CUDA graphs (uni_engine.py: one decode graph over every layer; generate.py,
sparkle: verify with per-token checkpoints, then the winning prefix committed),
through the C-ABI:

  - a captured decode step of every layer replays bit for bit like the eager
    calls, rows reaching their pool slots through state_idx, and matches the
    oracle layer by layer;
  - a captured verify of every layer followed by gdn_commit_accepted (one
    launch for all layers, the winner chosen on the device) leaves in each
    group's slot of every layer the oracle state after the winning path's
    accepted tokens; the winner equals the host rule (first longest accept
    length), an accept length of 0 commits nothing, and the result equals
    per-layer gdn_state_copy calls of the host-chosen checkpoint."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from gated_deltanet_recurrence_delta_gb300.stack import LayerStack
from tests.gpu_cases import ACTS, WEIGHTS, assert_out, assert_state, dims, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    build.build()
    gdn.load_library()


def _stack(shape, n_layers, n_slots, seed):
    g = torch.Generator().manual_seed(seed)
    ws_cpu = [I.weights(shape, g) for _ in range(n_layers)]
    st = I.states(shape, n_layers * n_slots, g, tail="randn")
    stack = LayerStack(shape, [{n: w[n].cuda() for n in WEIGHTS} for w in ws_cpu], n_slots)
    stack.state_pool.copy_(st["state"].view(stack.state_pool.shape))
    stack.conv_pool.copy_(st["conv_state"].view(stack.conv_pool.shape))
    return stack, ws_cpu, g


@pytest.mark.parametrize("shape", [I.TINY, I.Shape(nk=2, nv=4, dk=128, dv=128)])
def test_captured_decode_stack(oracle_mod, shape):
    L, n_slots, B = 3, 5, 3
    slots = [4, 0, 2]
    stack, ws_cpu, g = _stack(shape, L, n_slots, seed=110)
    S0, c0 = stack.state_pool.cpu(), stack.conv_pool.cpu()
    steps = [[I.activations(shape, B, 1, g) for _ in range(L)] for _ in range(2)]
    idx = torch.tensor(slots, dtype=torch.int32, device="cuda")

    # eager, on a copy of the pools
    eager = LayerStack(shape, stack.weights, n_slots)
    eager.state_pool.copy_(stack.state_pool)
    eager.conv_pool.copy_(stack.conv_pool)
    outs_e = []
    for acts in steps:
        out = torch.empty((L, B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
        eager.decode([{n: a[n].cuda() for n in ACTS} for a in acts], idx, out)
        outs_e.append(out)
    gdn.check_status()

    graph = stack.capture_decode(B)
    outs_g = []
    for acts in steps:
        for l in range(L):
            for n in ACTS:
                graph.acts[l][n].copy_(acts[l][n])
        graph.state_idx.copy_(idx)
        graph.replay()
        outs_g.append(graph.out.clone())
    torch.cuda.synchronize()
    gdn.check_status()
    for oe, og in zip(outs_e, outs_g):
        assert torch.equal(oe, og)
    assert torch.equal(stack.state_pool, eager.state_pool) and torch.equal(stack.conv_pool, eager.conv_pool)

    # the oracle, layer by layer, two tokens per row from the rows' slots
    for l in range(L):
        acts2 = {n: torch.cat([steps[0][l][n], steps[1][l][n]], 1) for n in ACTS}
        ref = oracle_layer(oracle_mod, shape, ws_cpu[l], acts2, c0[l][slots], S0[l][slots])
        assert_out(torch.cat([outs_g[0][l], outs_g[1][l]], 1), ref["out"], f"layer {l}")
        assert_state(stack.state_pool[l][slots], ref["state"], f"layer {l}")
        assert torch.equal(stack.conv_pool[l][slots].cpu().double(), torch.from_numpy(ref["conv_state"]))
    # slots no row names are untouched
    assert torch.equal(stack.state_pool[:, [1, 3]].cpu(), S0[:, [1, 3]])


@pytest.mark.parametrize("shape", [I.TINY, I.Shape(nk=2, nv=4, dk=128, dv=128)])
def test_captured_verify_and_fused_commit(oracle_mod, shape):
    L, n_slots, P, T = 3, 4, 4, 6
    groups = [3, 1]  # the pool slot of each group's sequence
    B = P * len(groups)
    stack, ws_cpu, g = _stack(shape, L, n_slots, seed=120)
    S0, c0 = stack.state_pool.cpu(), stack.conv_pool.cpu()
    acts = [I.activations(shape, B, T, g) for _ in range(L)]
    accept = torch.tensor([2, 5, 5, 1,  0, 0, 0, 0], dtype=torch.int32)  # group 1 accepts nothing
    graph = stack.capture_verify_commit(B, T, P)
    for l in range(L):
        for n in ACTS:
            graph.acts[l][n].copy_(acts[l][n])
    graph.state_idx.copy_(torch.tensor([s for s in groups for _ in range(P)], dtype=torch.int32))
    graph.accept_len.copy_(accept)
    graph.dst_slot.copy_(torch.tensor(groups, dtype=torch.int32))
    graph.replay()
    torch.cuda.synchronize()
    gdn.check_status()

    # the winner: the host rule of commit_tree_row, per group
    for gi in range(len(groups)):
        win, _ = gdn.commit_source_slot(accept[gi * P:(gi + 1) * P].tolist(), T)
        assert int(graph.winner[gi]) == gi * P + win
    # per-layer gdn_state_copy of the host-chosen checkpoint gives the same pools
    ref_S, ref_c = S0.clone().cuda(), c0.clone().cuda()
    for l in range(L):
        for gi, slot in enumerate(groups):
            win, src = gdn.commit_source_slot(accept[gi * P:(gi + 1) * P].tolist(), T)
            src_t = torch.tensor([-1 if src < 0 else gi * P * T + src], dtype=torch.int32, device="cuda")
            dst_t = torch.tensor([slot], dtype=torch.int32, device="cuda")
            gdn.state_copy(dims(shape, 1, 1, n_slots), graph.ckpt_state[l], graph.ckpt_conv[l], ref_S[l], ref_c[l],
                           src_t, dst_t, 1, B * T, n_slots)
    gdn.check_status()
    assert torch.equal(ref_S, stack.state_pool) and torch.equal(ref_c, stack.conv_pool)
    # against the oracle: the committed slot holds the state after the winner's accepted tokens
    for l in range(L):
        wi = 0 * P + 1  # group 0: rows 1 and 2 accept 5; the first wins
        La = int(accept[wi])
        a1 = {n: acts[l][n][wi:wi + 1, :La] for n in ACTS}
        ref = oracle_layer(oracle_mod, shape, ws_cpu[l], a1, c0[l][groups[0]:groups[0] + 1],
                           S0[l][groups[0]:groups[0] + 1])
        assert_state(stack.state_pool[l][groups[0]], ref["state"][0], f"layer {l}")
        assert torch.equal(stack.conv_pool[l][groups[0]].cpu().double(), torch.from_numpy(ref["conv_state"][0]))
        # group 1 (accept 0) and the slots no group names keep their states
        for sl in (groups[1], 0, 2):
            assert torch.equal(stack.state_pool[l][sl].cpu(), S0[l][sl])
            assert torch.equal(stack.conv_pool[l][sl].cpu(), c0[l][sl])
        # the verify outputs of every row from the shared slot
        for gi, slot in enumerate(groups):
            rows = slice(gi * P, (gi + 1) * P)
            ref = oracle_layer(oracle_mod, shape, ws_cpu[l], {n: acts[l][n][rows] for n in ACTS},
                               c0[l][[slot] * P], S0[l][[slot] * P])
            assert_out(graph.out[l][rows], ref["out"], f"layer {l} group {gi}")


def test_commit_accepted_bad_lengths_are_device_errors():
    """An accept length outside [0, T] or a slot outside the pool: recorded
    (GDN_ERR_INDEX), that group is not committed and its winner reads -1."""
    shape = I.TINY
    stack, _, _ = _stack(shape, 2, 2, seed=130)
    before = stack.state_pool.clone()
    B, T, P = 4, 3, 2
    ck = torch.randn((2, B, T, shape.nv, shape.dk, shape.dv), device="cuda")
    cc = torch.zeros((2, B, T, 3, shape.C), dtype=torch.bfloat16, device="cuda")
    acc = torch.tensor([1, 4, 2, 2], dtype=torch.int32, device="cuda")  # group 0 has a length > T
    dst = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    win = torch.zeros(2, dtype=torch.int32, device="cuda")
    stack.commit(P, acc, dst, ck, cc, win)
    with pytest.raises(gdn.GdnError) as e:
        gdn.check_status()
    assert e.value.name == "GDN_ERR_INDEX"
    assert win.tolist() == [-1, 2]
    assert torch.equal(stack.state_pool[:, 0], before[:, 0])
    for l in range(2):
        assert torch.equal(stack.state_pool[l, 1], ck[l, 2, 1])
    dst_bad = torch.tensor([0, 7], dtype=torch.int32, device="cuda")
    acc_ok = torch.tensor([1, 0, 0, 0], dtype=torch.int32, device="cuda")
    stack.commit(P, acc_ok, dst_bad, ck, cc, win)
    with pytest.raises(gdn.GdnError):
        gdn.check_status()
    assert win.tolist() == [0, -1]
    assert np.array_equal(stack.state_pool[:, 0].cpu().numpy(), ck[:, 0, 0].cpu().numpy())
