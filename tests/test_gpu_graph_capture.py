"""The C-ABI calls are asynchronous on the caller's stream and capturable into a
CUDA graph: a captured sequence (decode step, verify with checkpoints + commit,
a chunked prefill call) replayed from the graph gives exactly the results of
the same calls issued eagerly."""
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


def _case(shape, B, T_pre, T_ver, seed):
    d = I.decode_batch(seed=seed, B=B, shape=shape)
    g = torch.Generator().manual_seed(seed + 1)
    w = {n: dev(d[n]) for n in WEIGHTS}
    acts = {
        "pre": {n: dev(t) for n, t in I.activations(shape, B, T_pre, g).items()},
        "dec": {n: dev(t) for n, t in I.activations(shape, B, 1, g).items()},
        "ver": {n: dev(t) for n, t in I.activations(shape, B, T_ver, g).items()},
    }
    return d, w, acts


def _run(shape, B, T_pre, T_ver, w, acts, conv, S, out, ws):
    """prefill -> decode -> verify -> commit of row 0's last checkpoint, all on the current stream."""
    gdn.prefill_chunked(dims(shape, B, T_pre, B), inputs(w, acts["pre"]), conv, S, out["pre"], ws)
    gdn.decode_step(dims(shape, B, 1, B), inputs(w, acts["dec"]), conv, S, out["dec"])
    gdn.verify_with_checkpoints(dims(shape, B, T_ver, B), inputs(w, acts["ver"]), conv, S, out["ver"], out["cks"],
                                out["ckc"])
    gdn.state_copy(dims(shape, 1, 1, 1), out["cks"], out["ckc"], S, conv, out["src"], out["dst"], 1, B * T_ver, B)


@pytest.mark.parametrize("shape", [I.TINY, I.Shape(nk=2, nv=4, dk=128, dv=128)])
def test_captured_sequence_equals_eager(shape):
    B, T_pre, T_ver = 3, 130, 4
    d, w, acts = _case(shape, B, T_pre, T_ver, seed=90)

    def buffers():
        out = {
            "pre": torch.empty((B, T_pre, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda"),
            "dec": torch.empty((B, 1, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda"),
            "ver": torch.empty((B, T_ver, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda"),
            "cks": torch.empty((B, T_ver, shape.nv, shape.dk, shape.dv), dtype=torch.float32, device="cuda"),
            "ckc": torch.empty((B, T_ver, 3, shape.C), dtype=torch.bfloat16, device="cuda"),
            "src": torch.tensor([T_ver - 1], dtype=torch.int32, device="cuda"),
            "dst": torch.tensor([0], dtype=torch.int32, device="cuda"),
        }
        return out, dev(d["conv_state"]).clone(), dev(d["state"]).clone()

    ws = gdn.workspace(dims(shape, B, T_pre, B))
    out_e, conv_e, S_e = buffers()
    _run(shape, B, T_pre, T_ver, w, acts, conv_e, S_e, out_e, ws)
    gdn.check_status()

    out_g, conv_g, S_g = buffers()
    conv0, S0 = conv_g.clone(), S_g.clone()
    # warm-up outside the capture (first-use attribute setup), then restore the inputs
    _run(shape, B, T_pre, T_ver, w, acts, conv_g, S_g, out_g, ws)
    torch.cuda.synchronize()
    conv_g.copy_(conv0)
    S_g.copy_(S0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run(shape, B, T_pre, T_ver, w, acts, conv_g, S_g, out_g, ws)
    conv_g.copy_(conv0)
    S_g.copy_(S0)
    for n in out_g:
        if n not in ("src", "dst"):
            out_g[n].zero_()
    graph.replay()
    torch.cuda.synchronize()
    gdn.check_status()
    for n in ("pre", "dec", "ver", "cks", "ckc"):
        assert torch.equal(out_g[n], out_e[n]), n
    assert torch.equal(S_g, S_e) and torch.equal(conv_g, conv_e)
