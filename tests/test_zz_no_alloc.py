"""gdn_prefill_chunked_static_scratch -- the prefill for callers that cannot
allocate device memory (its scratch is a fixed array inside the library) --
gives the same results as gdn_prefill_chunked with a caller workspace, on two
calls in a row that continue the same rows. Collected last on purpose."""
import ctypes

import pytest
import torch

from gated_deltanet_recurrence_delta_gb300 import gdn
from gated_deltanet_recurrence_delta_gb300 import inputs as I
from tests.gpu_cases import ACTS, WEIGHTS, dev, dims, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    build.build()
    gdn.load_library()


@pytest.mark.parametrize("shape", [I.TINY, I.Shape(nk=2, nv=4, dk=128, dv=128)])
def test_static_scratch_matches_workspace_path(shape):
    """Both prefill paths (head size 32: CUDA cores; 128: tensor cores): the
    static scratch gives the results of a caller workspace, bit for bit."""
    d = I.decode_batch(seed=60, B=3, shape=shape)
    g = torch.Generator().manual_seed(61)
    calls = [I.activations(shape, 3, T, g) for T in (100, 37)]
    masks = [torch.ones(3, 100), torch.ones(3, 37)]
    masks[1][1, 20:] = 0  # a padded row in the second call
    w = {n: dev(d[n]) for n in WEIGHTS}
    ref_conv, ref_S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    new_conv, new_S = ref_conv.clone(), ref_S.clone()
    for acts, mask in zip(calls, masks):
        a = {n: dev(t) for n, t in acts.items()}
        m = dev(mask)
        T = a["q"].shape[1]
        dm = dims(shape, 3, T, 3)
        out_ref = torch.empty((3, T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
        out_new = torch.full_like(out_ref, 3.0)
        gdn.prefill_chunked(dm, inputs(w, a, mask=m), ref_conv, ref_S, out_ref, gdn.workspace(dm))
        gdn.prefill_chunked_static_scratch(dm, inputs(w, a, mask=m), new_conv, new_S, out_new)
        gdn.check_status()
        assert torch.equal(out_new, out_ref)
        assert torch.equal(new_S, ref_S)
        assert torch.equal(new_conv, ref_conv)


def test_static_scratch_rejects_oversized_calls():
    s = I.QWEN35_9B
    dm = dims(s, 1, 1 << 16, 1)   # 65536 tokens need far more than 64 MiB of scratch
    fake = gdn.Inputs(*([1 << 20] * 10 + [None, None, None]))
    lib = gdn.load_library()
    st = lib.gdn_prefill_chunked_static_scratch(ctypes.byref(dm), ctypes.byref(fake), 1 << 20, 1 << 20, 1 << 20, None)
    assert gdn.STATUS[st] == "GDN_ERR_WORKSPACE"
    assert "64 MiB" in gdn.last_error()
