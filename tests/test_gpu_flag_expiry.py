"""Expiry of the prefill chains' bounded flag waits, forced on a GPU without a
fault: a variant of the library is built with GDN_TEST_CHAIN_FLAGS_UNSET (a
state chain reads every chunk unit's flag as unset, as if no unit were ever
published) and a cap of 1024 polls. Nothing else changes in that build.

On a head-size-128 prefill of few chains (the chunk and state passes share one
grid and the chains wait on per-unit flags) every chain's first flag wait runs
out before it has issued any copy. The call must then report GDN_ERR_TIMEOUT
through the status word, return promptly, and leave every state, conv tail and
output of the call as it was. Packed rows, whose chains run in a separate
kernel after the chunk pass and wait on no flag, still match the oracle in the
same build.

The variant runs in a child process so that it never shares a process with
the in-tree library."""
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parent.parent

CHILD = textwrap.dedent(r"""
    import sys, time
    import torch
    sys.path.insert(0, sys.argv[2])
    from gated_deltanet_recurrence_delta_gb300 import gdn
    from gated_deltanet_recurrence_delta_gb300 import inputs as I
    from oracle import oracle
    from tests.gpu_cases import ACTS, WEIGHTS, assert_out, assert_state, dev, dims, inputs, oracle_layer

    gdn._lib = gdn.load_library(sys.argv[1])
    shape = I.Shape(nk=2, nv=4, dk=128, dv=128)
    d = I.decode_batch(seed=95, B=3, shape=shape)
    T = 130
    acts = I.activations(shape, 3, T, torch.Generator().manual_seed(96))
    w = {n: dev(d[n]) for n in WEIGHTS}
    dacts = {n: dev(a) for n, a in acts.items()}
    dm = dims(shape, 3, T, 3)
    ws = gdn.workspace(dm)

    # dense rows: 3 rows x 4 value heads = 12 chains over 36 chunk units -> one grid
    times = []
    for rep in range(2):
        conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
        out = torch.full((3, T, shape.nv, shape.dv), 7.0, dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        gdn.prefill_chunked(dm, inputs(w, dacts), conv, S, out, ws)
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
        try:
            gdn.check_status()
            raise SystemExit("expected GDN_ERR_TIMEOUT, the call reported OK")
        except gdn.GdnError as e:
            assert e.name == "GDN_ERR_TIMEOUT", e.name
        assert torch.equal(S.cpu(), d["state"]), "a stopped chain wrote its state"
        assert torch.equal(conv.cpu(), d["conv_state"]), "a stopped chain wrote its conv tail"
        assert bool(torch.all(out.float() == 7.0)), "a stopped chain's outputs were written"
    # the second call (module loaded, caches warm): every chain gave up after its
    # 1024 polls and left; no second wait ran to its own bound
    assert times[1] < 0.25, f"the call took {times[1]:.3f} s"

    # packed rows: the chains run in their own kernel and read no flag
    cu = torch.tensor([0, T, 2 * T, 3 * T], dtype=torch.int32)
    pacts = {n: a.reshape(1, 3 * T, -1).contiguous() for n, a in acts.items()}
    conv, S = dev(d["conv_state"]).clone(), dev(d["state"]).clone()
    out = torch.empty((1, 3 * T, shape.nv, shape.dv), dtype=torch.bfloat16, device="cuda")
    pdm = dims(shape, 3, 3 * T, 3)
    gdn.prefill_chunked(pdm, inputs(w, {n: dev(a) for n, a in pacts.items()}, cu=dev(cu)), conv, S, out,
                        gdn.workspace(pdm, packed=True))
    gdn.check_status()
    oracle.build()
    ref = oracle_layer(oracle, shape, d, acts, d["conv_state"], d["state"])
    assert_out(out.reshape(3, T, shape.nv, shape.dv), ref["out"])
    assert_state(S, ref["state"])
    assert torch.equal(conv.cpu().double(), torch.from_numpy(ref["conv_state"]))
    print("flag expiry ok", ["%.4f" % t for t in times])
""")


def test_chain_flag_wait_expiry_leaves_heads_whole(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_deltanet_recurrence_delta_gb300 import build
    lib = build.build(force=True, out_dir=tmp_path / "flag_expiry_build",
                      defines=("GDN_TEST_CHAIN_FLAGS_UNSET", "GDN_FLAG_WAIT_CAP=1024"))
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    r = subprocess.run([sys.executable, str(script), str(lib), str(ROOT)], capture_output=True, text=True,
                       timeout=600, cwd=str(ROOT))
    assert r.returncode == 0, f"child failed:\n{r.stdout}\n{r.stderr}"
    assert "flag expiry ok" in r.stdout
