"""GPU parity of gdn_decode_step, gdn_verify_with_checkpoints and gdn_state_copy
against the fp64 oracle, through the C-ABI."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from tests.gpu_cases import (ACTS, WEIGHTS, assert_out, assert_state, dev, dims, inputs, max_abs,
                             oracle_layer)

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


def _acts(d, sl=slice(None)):
    return {n: dev(d[n][:, sl].contiguous()) for n in ACTS}


def _decode(shape, w, acts, conv, S, mask=None, state_idx=None, n_slots=None):
    B = acts["q"].shape[0]
    out = torch.empty((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    inp = inputs(w, acts, mask=mask, state_idx=state_idx)
    gdn.decode_step(dims(shape, B, 1, n_slots or conv.shape[0]), inp, conv, S, out)
    return out


def test_decode_batch_qwen_layout(oracle_mod):
    """64 rows, 16/32 heads, d=128, one token, random state and conv tail."""
    d = I.decode_batch(seed=1)
    s = d["shape"]
    w, acts = _wd(d), _acts(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _decode(s, w, acts, conv, S)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, s, d, d, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


@pytest.mark.parametrize("B", [1, 200])
def test_decode_row_counts(oracle_mod, B):
    """The 16/32-head d=128 layer with 1 row (16 units: most CTAs have none)
    and with 200 rows (3200 (row, key head) units over one CTA per SM: each
    CTA streams ~42 heads through its three-stage copy ring, many wraps of the
    ring's phases, and the last units are ragged)."""
    d = I.decode_batch(seed=31, B=B)
    s = d["shape"]
    w, acts = _wd(d), _acts(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _decode(s, w, acts, conv, S)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, s, d, d, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


@pytest.mark.parametrize("shape", [I.TINY, I.Shape(nk=4, nv=8, dk=64, dv=64), I.Shape(nk=2, nv=2, dk=128, dv=128),
                                   I.Shape(nk=1, nv=4, dk=128, dv=128)])
def test_decode_head_sizes(oracle_mod, shape):
    d = I.decode_batch(seed=11, B=5, shape=shape)
    w, acts = _wd(d), _acts(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = _decode(shape, w, acts, conv, S)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, shape, d, d, d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))


def test_decode_mask_and_state_pool(oracle_mod):
    """Rows map to pool slots through state_idx; a row with mask 0 is left
    untouched bit for bit and gets zero output; unused slots are untouched."""
    shape = I.TINY
    d = I.decode_batch(seed=12, B=4, shape=shape)
    pool = I.states(shape, 6, torch.Generator().manual_seed(5))
    idx = torch.tensor([4, 0, 2, 5], dtype=torch.int32)
    mask = torch.tensor([1.0, 0.0, 1.0, 0.0])
    w, acts = _wd(d), _acts(d)
    conv0, S0 = pool["conv_state"], pool["state"]
    conv, S = dev(conv0).clone(), dev(S0).clone()
    out = _decode(shape, w, acts, conv, S, mask=dev(mask), state_idx=dev(idx), n_slots=6)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, shape, d, d, conv0[idx.long()], S0[idx.long()], mask=mask[:, None])
    for r in range(4):
        slot = int(idx[r])
        if mask[r] == 1:
            assert_out(out[r], ref["out"][r])
            assert_state(S[slot], ref["state"][r])
            assert torch.equal(conv[slot].cpu().double(), torch.from_numpy(ref["conv_state"][r]))
        else:
            assert torch.equal(S[slot].cpu(), S0[slot]) and torch.equal(conv[slot].cpu(), conv0[slot])
            assert torch.count_nonzero(out[r]) == 0
    for slot in (1, 3):
        assert torch.equal(S[slot].cpu(), S0[slot]) and torch.equal(conv[slot].cpu(), conv0[slot])


def _host_mapped(t):
    """True when the pinned host tensor t is mapped into the device's address
    space at its own address (driver pointer attributes: memory type = host,
    device pointer = the host pointer)."""
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    cu.cuPointerGetAttribute.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64]
    mt, dp = ctypes.c_uint(0), ctypes.c_uint64(0)
    CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_DEVICE_POINTER, CU_MEMORYTYPE_HOST = 2, 3, 1
    if cu.cuPointerGetAttribute(ctypes.byref(mt), CU_POINTER_ATTRIBUTE_MEMORY_TYPE, t.data_ptr()) != 0:
        return False
    if cu.cuPointerGetAttribute(ctypes.byref(dp), CU_POINTER_ATTRIBUTE_DEVICE_POINTER, t.data_ptr()) != 0:
        return False
    return mt.value == CU_MEMORYTYPE_HOST and dp.value == t.data_ptr()


def test_decode_zero_copy_host_activations(oracle_mod):
    """The activations and the output rows in pinned host memory (the kernel
    reads and writes them across the host link): bit for bit the call on
    device buffers, and the oracle's result."""
    d = I.decode_batch(seed=21, B=64)
    s = d["shape"]
    w, acts = _wd(d), _acts(d)
    hacts = {n: d[n].contiguous().pin_memory() for n in ACTS}
    hout = torch.zeros((64, 1, s.nv, s.dv), dtype=torch.bfloat16).pin_memory()
    if not all(_host_mapped(t) for t in list(hacts.values()) + [hout]):
        pytest.skip("pinned host memory is not mapped at its own address on this system")
    conv_d, S_d = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    conv_h, S_h = conv_d.clone(), S_d.clone()
    out_d = _decode(s, w, acts, conv_d, S_d)
    gdn.decode_step(dims(s, 64, 1, 64), inputs(w, hacts), conv_h, S_h, hout)
    torch.cuda.synchronize()
    gdn.check_status()
    assert torch.equal(hout, out_d.cpu())
    assert torch.equal(S_h, S_d) and torch.equal(conv_h, conv_d)
    ref = oracle_layer(oracle_mod, s, d, d, d["conv_state"], d["state"])
    assert_out(hout, ref["out"])


@pytest.mark.parametrize("shape,T", [(I.TINY, 8), (I.QWEN35_9B, 8), (I.Shape(nk=1, nv=4, dk=128, dv=128), 8),
                                     (I.Shape(nk=1, nv=4, dk=128, dv=128), 1), (I.Shape(nk=1, nv=4, dk=128, dv=128), 2),
                                     (I.Shape(nk=1, nv=4, dk=128, dv=128), 3), (I.Shape(nk=1, nv=4, dk=128, dv=128), 5),
                                     (I.Shape(nk=1, nv=4, dk=128, dv=128), 7)])
def test_verify_checkpoints_equal_decode_steps_bitwise(shape, T):
    """Verify checkpoint t == the state after t+1 decode steps, bit for bit; the
    conv checkpoint == the decoded conv tail; the outputs are identical. Token
    counts below 8 leave warps of the head-size-128 kernel without a token, and
    up to 3 tokens every convolution reads the saved tail."""
    B = 2
    d = I.verify_paths(seed=21, P=B, K=T, shape=shape)
    w = _wd(d)
    acts = _acts(d)
    conv0 = dev(d["conv_state"]).expand(B, -1, -1).contiguous()
    S0 = dev(d["state"]).expand(B, -1, -1, -1).contiguous()
    out_v = torch.empty((B, T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    ck_s = torch.empty((B, T, shape.nv, shape.dk, shape.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.empty((B, T, 3, shape.C), dtype=torch.bfloat16, device="cuda")
    gdn.verify_with_checkpoints(dims(shape, B, T, B), inputs(w, acts), conv0, S0, out_v, ck_s, ck_c)
    conv, S = conv0.clone(), S0.clone()
    for t in range(T):
        a_t = {n: acts[n][:, t:t + 1].contiguous() for n in ACTS}
        out = _decode(shape, w, a_t, conv, S)
        assert torch.equal(out[:, 0], out_v[:, t])
        assert torch.equal(S, ck_s[:, t]), f"state checkpoint {t} differs"
        assert torch.equal(conv, ck_c[:, t]), f"conv checkpoint {t} differs"
    gdn.check_status()


def test_verify_rows_over_a_state_pool(oracle_mod):
    """Verify rows read their states from pool slots through state_idx: rows 0
    and 3 share slot 4, rows 1 and 2 read slots 0 and 6 (out of order, 7
    slots). Outputs and every checkpoint against the oracle from each row's
    slot; the pool is read only."""
    shape, B, T, n_slots = I.Shape(nk=2, nv=4, dk=128, dv=128), 4, 6, 7
    idx = torch.tensor([4, 0, 6, 4], dtype=torch.int32)
    g = torch.Generator().manual_seed(180)
    pool = I.states(shape, n_slots, g)
    d = I.decode_batch(seed=181, B=B, shape=shape)
    acts = I.activations(shape, B, T, g)
    w = _wd(d)
    conv, S = dev(pool["conv_state"]).clone(), dev(pool["state"]).clone()
    out = torch.empty((B, T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    ck_s = torch.empty((B, T, shape.nv, shape.dk, shape.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.empty((B, T, 3, shape.C), dtype=torch.bfloat16, device="cuda")
    gdn.verify_with_checkpoints(dims(shape, B, T, n_slots), inputs(w, {n: dev(a) for n, a in acts.items()},
                                                                   state_idx=dev(idx)), conv, S, out, ck_s, ck_c)
    gdn.check_status()
    il = idx.long()
    ref = oracle_layer(oracle_mod, shape, d, acts, pool["conv_state"][il], pool["state"][il], checkpoints=True)
    assert_out(out, ref["out"])
    for r in range(B):
        for t in range(T):
            assert_state(ck_s[r, t], ref["ckpt_state"][r, t], f"ckpt[{r},{t}]")
    assert torch.equal(ck_c.cpu().double(), torch.from_numpy(ref["ckpt_conv"]))
    assert torch.equal(S.cpu(), pool["state"]) and torch.equal(conv.cpu(), pool["conv_state"])


def test_verify_paths_and_commit(oracle_mod):
    """8 paths x 8 draft tokens from one shared state (state_idx = 0 for every
    row); commit the winner's checkpoint at its accept length."""
    d = I.verify_paths(seed=3)
    s = d["shape"]
    P, K = 8, 8
    w, acts = _wd(d), _acts(d)
    conv, S = dev(d["conv_state"]), dev(d["state"])
    idx = torch.zeros(P, dtype=torch.int32, device="cuda")
    out = torch.empty((P, K, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
    ck_s = torch.empty((P, K, s.nv, s.dk, s.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.empty((P, K, 3, s.C), dtype=torch.bfloat16, device="cuda")
    gdn.verify_with_checkpoints(dims(s, P, K, 1), inputs(w, acts, state_idx=idx), conv, S, out, ck_s, ck_c)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, s, d, d, d["conv_state"].expand(P, -1, -1), d["state"].expand(P, -1, -1, -1),
                       checkpoints=True)
    assert_out(out, ref["out"])
    for p in range(P):
        for t in range(K):
            assert_state(ck_s[p, t], ref["ckpt_state"][p, t], f"ckpt[{p},{t}]")
    assert torch.equal(ck_c.cpu().double(), torch.from_numpy(ref["ckpt_conv"]))
    # the shared state is read only
    assert torch.equal(S.cpu(), d["state"]) and torch.equal(conv.cpu(), d["conv_state"])

    # commit: winner = first path with the longest accept length (ties -> lower index)
    L = d["accept_len"].tolist()
    win = int(np.argmax(L))
    assert L[win] == max(L) and all(l < L[win] for l in L[:win])
    src = torch.tensor([win * K + L[win] - 1 if L[win] > 0 else -1], dtype=torch.int32, device="cuda")
    dst = torch.zeros(1, dtype=torch.int32, device="cuda")
    S_pool, conv_pool = S.clone(), conv.clone()
    gdn.state_copy(dims(s, 1, 1, 1), ck_s, ck_c, S_pool, conv_pool, src, dst, 1, P * K, 1)
    gdn.check_status()
    if L[win] > 0:
        assert torch.equal(S_pool[0], ck_s[win, L[win] - 1])
        assert torch.equal(conv_pool[0], ck_c[win, L[win] - 1])
    else:
        assert torch.equal(S_pool, S) and torch.equal(conv_pool, conv)


def test_commit_accept_zero_and_errors():
    """src_slot -1 commits nothing; an out-of-range slot is a recorded device error."""
    s = I.TINY
    g = torch.Generator().manual_seed(3)
    src = I.states(s, 4, g)
    dstp = I.states(s, 2, g)
    S_src, c_src = dev(src["state"]), dev(src["conv_state"])
    S_dst, c_dst = dev(dstp["state"]).clone(), dev(dstp["conv_state"]).clone()
    ss = torch.tensor([-1, 3], dtype=torch.int32, device="cuda")
    ds = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    gdn.state_copy(dims(s, 1, 1, 1), S_src, c_src, S_dst, c_dst, ss, ds, 2, 4, 2)
    gdn.check_status()
    assert torch.equal(S_dst[0].cpu(), dstp["state"][0]) and torch.equal(c_dst[0].cpu(), dstp["conv_state"][0])
    assert torch.equal(S_dst[1], S_src[3]) and torch.equal(c_dst[1], c_src[3])
    bad = torch.tensor([4], dtype=torch.int32, device="cuda")
    gdn.state_copy(dims(s, 1, 1, 1), S_src, c_src, S_dst, c_dst, bad, ds[:1], 1, 4, 2)
    with pytest.raises(gdn.GdnError) as e:
        gdn.check_status()
    assert e.value.name == "GDN_ERR_INDEX"


def test_verify_padding_repeats_last_checkpoint(oracle_mod):
    s = I.TINY
    B, T = 2, 8
    d = I.verify_paths(seed=22, P=B, K=T, shape=s)
    mask = torch.zeros((B, T))
    mask[0, :5] = 1
    mask[1, :0] = 1  # a row with no real token
    w, acts = _wd(d), _acts(d)
    conv0 = dev(d["conv_state"]).expand(B, -1, -1).contiguous()
    S0 = dev(d["state"]).expand(B, -1, -1, -1).contiguous()
    out = torch.full((B, T, s.nv, s.dv), 7.0, dtype=torch.bfloat16, device="cuda")
    ck_s = torch.empty((B, T, s.nv, s.dk, s.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.empty((B, T, 3, s.C), dtype=torch.bfloat16, device="cuda")
    gdn.verify_with_checkpoints(dims(s, B, T, B), inputs(w, acts, mask=dev(mask)), conv0, S0, out, ck_s, ck_c)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, s, d, d, conv0.cpu(), S0.cpu(), mask=mask, checkpoints=True)
    assert_out(out[0, :5], ref["out"][0, :5])
    assert torch.count_nonzero(out[0, 5:]) == 0 and torch.count_nonzero(out[1]) == 0
    for t in range(T):
        assert_state(ck_s[0, t], ref["ckpt_state"][0, t])
        assert torch.equal(ck_s[1, t], S0[1])
    for t in range(5, T):
        assert torch.equal(ck_s[0, t], ck_s[0, 4])
    assert torch.equal(ck_c.cpu().double(), torch.from_numpy(ref["ckpt_conv"]))


def test_device_errors_skip_rows():
    """A non-prefix mask row and an out-of-range slot are recorded and the rows
    skipped (state untouched)."""
    s = I.TINY
    d = I.verify_paths(seed=23, P=2, K=4, shape=s)
    w, acts = _wd(d), _acts(d)
    conv0 = dev(d["conv_state"]).expand(2, -1, -1).contiguous()
    S0 = dev(d["state"]).expand(2, -1, -1, -1).contiguous()
    mask = torch.tensor([[1.0, 0.0, 1.0, 0.0], [1.0, 1.0, 1.0, 1.0]], device="cuda")
    out = torch.empty((2, 4, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
    ck_s = torch.zeros((2, 4, s.nv, s.dk, s.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.zeros((2, 4, 3, s.C), dtype=torch.bfloat16, device="cuda")
    gdn.verify_with_checkpoints(dims(s, 2, 4, 2), inputs(w, acts, mask=mask), conv0, S0, out, ck_s, ck_c)
    with pytest.raises(gdn.GdnError) as e:
        gdn.check_status()
    assert e.value.name == "GDN_ERR_MASK"
    assert torch.count_nonzero(ck_s[0]) == 0 and torch.count_nonzero(ck_s[1]) > 0
    gdn.check_status()  # cleared
    a1 = {n: acts[n][:, :1].contiguous() for n in ACTS}
    conv, S = conv0.clone(), S0.clone()
    idx = torch.tensor([0, 7], dtype=torch.int32, device="cuda")
    _decode(s, w, a1, conv, S, state_idx=idx, n_slots=2)
    with pytest.raises(gdn.GdnError) as e:
        gdn.check_status()
    assert e.value.name == "GDN_ERR_INDEX"


def test_tiny_layer_prefill_decode_verify(oracle_mod):
    """The tiny layer end to end: prefill 64 tokens, 8 decode steps, then a
    verify of 8 tokens, each against the oracle continuing the same sequence."""
    d = I.tiny_layer(0)
    s = d["shape"]
    w = _wd(d)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    pre = {n: dev(d["prefill"][n]) for n in ACTS}
    out = torch.empty((1, 64, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
    dm = dims(s, 1, 64, 1)
    ws = gdn.workspace(dm)
    gdn.prefill_chunked(dm, inputs(w, pre), conv, S, out, ws)
    gdn.check_status()
    ref = oracle_layer(oracle_mod, s, d, d["prefill"], d["conv_state"], d["state"])
    assert_out(out, ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))
    o_conv, o_S = ref["conv_state"], ref["state"]
    for t in range(8):
        a_t = {n: dev(d["decode"][n][:, t:t + 1].contiguous()) for n in ACTS}
        o = _decode(s, w, a_t, conv, S)
        r = oracle_layer(oracle_mod, s, d, {n: d["decode"][n][:, t:t + 1] for n in ACTS},
                         torch.from_numpy(o_conv), torch.from_numpy(o_S))
        o_conv, o_S = r["conv_state"], r["state"]
        assert_out(o, r["out"])
    assert_state(S, o_S)
    va = {n: dev(d["verify"][n]) for n in ACTS}
    out_v = torch.empty((1, 8, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
    ck_s = torch.empty((1, 8, s.nv, s.dk, s.dv), dtype=torch.float32, device="cuda")
    ck_c = torch.empty((1, 8, 3, s.C), dtype=torch.bfloat16, device="cuda")
    gdn.verify_with_checkpoints(dims(s, 1, 8, 1), inputs(w, va), conv, S, out_v, ck_s, ck_c)
    gdn.check_status()
    r = oracle_layer(oracle_mod, s, d, d["verify"], torch.from_numpy(o_conv), torch.from_numpy(o_S),
                     checkpoints=True)
    assert_out(out_v, r["out"])
    for t in range(8):
        assert_state(ck_s[0, t], r["ckpt_state"][0, t])


def test_copy_overlapped_bytes():
    """One gdn_copy_overlapped call with an upload from pinned host memory, a
    read-back into it and a device-to-device copy, of ragged sizes: every
    destination equals its source byte for byte, and the bytes around the
    destinations are untouched."""
    g = torch.Generator().manual_seed(190)
    sizes = [16, 4112, 1581056]
    srcs_h = [torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g).pin_memory() for n in sizes]
    if not all(_host_mapped(t) for t in srcs_h):
        pytest.skip("pinned host memory is not mapped at its own address on this system")
    dev_src = torch.randint(0, 256, (sizes[2],), dtype=torch.uint8, generator=g).cuda()
    pad = 64
    up = torch.full((sizes[2] + 2 * pad,), 7, dtype=torch.uint8, device="cuda")
    down = torch.full((sizes[1] + 2 * pad,), 9, dtype=torch.uint8).pin_memory()
    d2d = torch.full((sizes[2] + 2 * pad,), 5, dtype=torch.uint8, device="cuda")
    gdn.copy_overlapped([(up[pad:].data_ptr(), srcs_h[2], sizes[2]),
                         (down[pad:].data_ptr(), dev_src[:sizes[1]], sizes[1]),
                         (d2d[pad:].data_ptr(), dev_src, sizes[2]),
                         (up.data_ptr(), srcs_h[0], 0)])
    torch.cuda.synchronize()
    gdn.check_status()
    assert torch.equal(up[pad:pad + sizes[2]].cpu(), srcs_h[2])
    assert torch.equal(down[pad:pad + sizes[1]], dev_src[:sizes[1]].cpu())
    assert torch.equal(d2d[pad:pad + sizes[2]], dev_src)
    assert (up[:pad] == 7).all() and (up[pad + sizes[2]:] == 7).all()
    assert (down[:pad] == 9).all() and (down[pad + sizes[1]:] == 9).all()
    assert (d2d[:pad] == 5).all() and (d2d[pad + sizes[2]:] == 5).all()


def test_decode_loop_staged_through_overlapped_copies():
    """A 6-step decode loop fed from pinned host memory, one state carried
    from step to step: step i+1's activations go up and step i-1's output rows
    come down in one gdn_copy_overlapped call queued right after step i (two
    device input sets, two device output sets). Every step's rows on the host
    and the final state and conv tail equal 6 plain steps on device inputs,
    bit for bit."""
    shape, B, K = I.Shape(nk=2, nv=4, dk=128, dv=128), 8, 6
    d = I.decode_batch(seed=191, B=B, shape=shape)
    w = _wd(d)
    steps = [I.activations(shape, B, 1, torch.Generator().manual_seed(192 + i)) for i in range(K)]
    host_in = [{n: s[n].contiguous().pin_memory() for n in ACTS} for s in steps]
    host_out = [torch.zeros((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16).pin_memory() for _ in range(K)]
    if not all(_host_mapped(t) for h in host_in for t in h.values()):
        pytest.skip("pinned host memory is not mapped at its own address on this system")
    dev_in = [{n: torch.empty_like(steps[0][n], device="cuda") for n in ACTS} for _ in range(2)]
    dev_out = [torch.empty((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dm = dims(shape, B, 1, B)
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()

    def up(i):
        return [(dev_in[i % 2][n], host_in[i][n], host_in[i][n].numel() * host_in[i][n].element_size())
                for n in ACTS]

    def down(i):
        return [(host_out[i], dev_out[i % 2], host_out[i].numel() * 2)]

    gdn.copy_overlapped(up(0))
    for i in range(K):
        gdn.decode_step(dm, inputs(w, dev_in[i % 2]), conv, S, dev_out[i % 2])
        gdn.copy_overlapped((up(i + 1) if i + 1 < K else []) + (down(i - 1) if i >= 1 else []))
    host_out[K - 1].copy_(dev_out[(K - 1) % 2])  # the last step's rows, once the stream has passed it
    torch.cuda.synchronize()
    gdn.check_status()
    conv_r, S_r = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    for i in range(K):
        out_r = _decode(shape, w, {n: dev(steps[i][n]) for n in ACTS}, conv_r, S_r)
        assert torch.equal(host_out[i], out_r.cpu()), f"step {i}"
    assert torch.equal(S, S_r) and torch.equal(conv, conv_r)
