"""GPU parity of gdn_decode_step_mxfp8 (the decode step with its token channels
q / k / v / z in MXFP8: e4m3 elements, one power-of-two E8M0 scale per 32
channels), through the C-ABI:

  - bit for bit equal to gdn_decode_step on the dequantized inputs (outputs,
    fp32 state and bf16 conv tail): everything after dequantization is the
    bf16 path's arithmetic;
  - against the oracle on the dequantized inputs within the spec bars;
  - against the oracle on the original bf16 inputs (before quantization): the
    error FP8 itself brings (e4m3 keeps 4 significant bits, so each input
    moves by up to ~6%), recorded, with loose sanity bounds on the relative
    Frobenius errors of the outputs and of the state after the token."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from tests.gpu_cases import ACTS, WEIGHTS, assert_out, assert_state, dev, dims, inputs, oracle_layer, record, rel_fro

pytestmark = pytest.mark.gpu

MX = ("q", "k", "v", "z")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    build.build()
    gdn.load_library()


def dequant(e, s, block=32):
    """The value an MXFP8 element stands for: e4m3 times 2^(scale - 127)."""
    f = e.view(torch.float8_e4m3fn).float()
    sc = torch.exp2(s.float() - 127.0)
    return (f.reshape(*f.shape[:-1], -1, block) * sc.unsqueeze(-1)).reshape(f.shape)


@pytest.mark.parametrize("shape,B", [(I.QWEN35_9B, 16), (I.TINY, 3), (I.Shape(nk=1, nv=4, dk=64, dv=64), 2)])
def test_mxfp8_decode(oracle_mod, shape, B):
    d = I.decode_batch(seed=140 + B, B=B, shape=shape)
    enc = {n: I.mxfp8(d[n]) for n in MX}
    deq = {n: dequant(*enc[n]).to(torch.bfloat16) for n in MX}
    for n in MX:  # every dequantized element is exact in bf16
        assert torch.equal(deq[n].float(), dequant(*enc[n]))
    acts_deq = {**{n: d[n] for n in ACTS}, **deq}
    w = {n: dev(d[n]) for n in WEIGHTS}
    dm = dims(shape, B, 1, B)

    # the MXFP8 call
    conv8, S8 = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out8 = torch.empty((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    mx = {n: (dev(enc[n][0]), dev(enc[n][1])) for n in MX}
    inp8 = gdn.make_inputs_mxfp8(mx["q"][0], mx["k"][0], mx["v"][0], mx["z"][0], mx["q"][1], mx["k"][1],
                                 mx["v"][1], mx["z"][1], dev(d["a"]), dev(d["b"]), w["A_log"], w["dt_bias"],
                                 w["conv_w"], w["norm_w"])
    gdn.decode_step_mxfp8(dm, inp8, conv8, S8, out8)
    # the bf16 call on the dequantized inputs
    convb, Sb = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    outb = torch.empty_like(out8)
    gdn.decode_step(dm, inputs(w, {n: dev(a) for n, a in acts_deq.items()}), convb, Sb, outb)
    gdn.check_status()
    assert torch.equal(out8, outb) and torch.equal(S8, Sb) and torch.equal(conv8, convb)

    # the oracle on the dequantized inputs: the spec bars
    ref = oracle_layer(oracle_mod, shape, d, acts_deq, d["conv_state"], d["state"])
    assert_out(out8, ref["out"])
    assert_state(S8, ref["state"])
    assert torch.equal(conv8.cpu().double(), torch.from_numpy(ref["conv_state"]))

    # the oracle on the original bf16 inputs: what FP8 itself costs
    ref0 = oracle_layer(oracle_mod, shape, d, d, d["conv_state"], d["state"])
    e_out = rel_fro(out8, ref0["out"])
    e_state = rel_fro(S8, ref0["state"])
    record("fp8_vs_bf16_inputs_out_rel_fro", e_out)
    record("fp8_vs_bf16_inputs_state_rel_fro", e_state)
    assert e_out <= 0.15, f"outputs {e_out:.3e} off the bf16-input result (relative Frobenius)"
    assert e_state <= 0.1, f"state {e_state:.3e} off the bf16-input result (relative Frobenius)"
    assert np.isfinite(e_out) and np.isfinite(e_state)


def test_mxfp8_decode_masked_rows_and_state_pool():
    """The benchmark's size (64 rows, 16/32 heads, d=128) with two masked rows
    and each row's state in a pool slot of its own (a permutation of 70 slots):
    the MXFP8 step equals the bf16 step on the dequantized inputs bit for bit,
    masked rows and unused slots untouched."""
    shape, B, n_slots = I.QWEN35_9B, 64, 70
    d = I.decode_batch(seed=147, B=B, shape=shape)
    enc = {n: I.mxfp8(d[n]) for n in MX}
    deq = {n: dequant(*enc[n]).to(torch.bfloat16) for n in MX}
    acts_deq = {**{n: d[n] for n in ACTS}, **deq}
    w = {n: dev(d[n]) for n in WEIGHTS}
    g = torch.Generator().manual_seed(148)
    slots = torch.randperm(n_slots, generator=g)[:B].to(torch.int32)
    mask = torch.ones(B)
    mask[[5, 40]] = 0.0
    pool_S = torch.randn((n_slots, shape.nv, shape.dk, shape.dv), generator=g) * 0.1
    pool_c = (torch.randn((n_slots, 3, shape.C), generator=g)).to(torch.bfloat16)
    dm = dims(shape, B, 1, n_slots)
    conv8, S8 = dev(pool_c).clone(), dev(pool_S).clone()
    out8 = torch.empty((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    mx = {n: (dev(enc[n][0]), dev(enc[n][1])) for n in MX}
    inp8 = gdn.make_inputs_mxfp8(mx["q"][0], mx["k"][0], mx["v"][0], mx["z"][0], mx["q"][1], mx["k"][1],
                                 mx["v"][1], mx["z"][1], dev(d["a"]), dev(d["b"]), w["A_log"], w["dt_bias"],
                                 w["conv_w"], w["norm_w"], mask=dev(mask), state_idx=dev(slots))
    gdn.decode_step_mxfp8(dm, inp8, conv8, S8, out8)
    convb, Sb = dev(pool_c).clone(), dev(pool_S).clone()
    outb = torch.empty_like(out8)
    gdn.decode_step(dm, inputs(w, {n: dev(a) for n, a in acts_deq.items()}, mask=dev(mask), state_idx=dev(slots)),
                    convb, Sb, outb)
    gdn.check_status()
    assert torch.equal(out8, outb) and torch.equal(S8, Sb) and torch.equal(conv8, convb)
    untouched = sorted(set(range(n_slots)) - set(slots.tolist())) + [int(slots[5]), int(slots[40])]
    for s_ in untouched:
        assert torch.equal(S8[s_].cpu(), pool_S[s_]) and torch.equal(conv8[s_].cpu(), pool_c[s_]), f"slot {s_}"
    assert all(not torch.equal(S8[int(slots[r])].cpu(), pool_S[int(slots[r])]) for r in (0, 1, 63))
    assert torch.count_nonzero(out8[[5, 40]]) == 0


def test_mxfp8_every_code_at_several_scales():
    """Every finite e4m3 code (254 of the 256 bytes; S.1111.111 is NaN), with
    block scales from 2^-117 to 2^7, so that every dequantized value, from the
    smallest subnormal code to 448, lands in bf16's normal range: the MXFP8
    step equals the bf16 step on the dequantized inputs bit for bit. This pins
    the kernel's e4m3 decoding (subnormals, the sign, the largest code) and its
    scaling against torch's float8_e4m3fn conversion."""
    shape, B = I.QWEN35_9B, 4
    d = I.decode_batch(seed=149, B=B, shape=shape)
    codes = torch.tensor([c for c in range(256) if c & 0x7F != 0x7F], dtype=torch.uint8)
    scales = torch.tensor([10, 100, 127, 134, 120], dtype=torch.uint8)  # 2^(s - 127)
    enc = {}
    for i, n in enumerate(MX):
        numel = d[n].numel()
        e = codes[(torch.arange(numel) + 37 * i) % codes.numel()].reshape(d[n].shape)
        s = scales[(torch.arange(numel // 32) + i) % scales.numel()].reshape(*d[n].shape[:-1], -1)
        enc[n] = (e, s)
    assert all(set(enc[n][0].flatten().tolist()) == set(codes.tolist()) for n in MX)
    deq = {n: dequant(*enc[n]).to(torch.bfloat16) for n in MX}
    for n in MX:  # every dequantized value is exact in bf16 and normal (or zero)
        f = dequant(*enc[n])
        assert torch.equal(deq[n].float(), f)
        nz = f[f != 0].abs()
        assert float(nz.min()) >= 2.0 ** -126 and float(nz.max()) <= 448.0 * 2.0 ** 7
    acts_deq = {**{n: d[n] for n in ACTS}, **deq}
    w = {n: dev(d[n]) for n in WEIGHTS}
    dm = dims(shape, B, 1, B)
    conv8, S8 = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out8 = torch.empty((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    mx = {n: (dev(enc[n][0]), dev(enc[n][1])) for n in MX}
    inp8 = gdn.make_inputs_mxfp8(mx["q"][0], mx["k"][0], mx["v"][0], mx["z"][0], mx["q"][1], mx["k"][1],
                                 mx["v"][1], mx["z"][1], dev(d["a"]), dev(d["b"]), w["A_log"], w["dt_bias"],
                                 w["conv_w"], w["norm_w"])
    gdn.decode_step_mxfp8(dm, inp8, conv8, S8, out8)
    convb, Sb = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    outb = torch.empty_like(out8)
    gdn.decode_step(dm, inputs(w, {n: dev(a) for n, a in acts_deq.items()}), convb, Sb, outb)
    gdn.check_status()
    assert torch.isfinite(out8.float()).all() and torch.isfinite(S8).all()
    assert torch.equal(out8, outb) and torch.equal(S8, Sb) and torch.equal(conv8, convb)
