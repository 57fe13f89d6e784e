"""The C-ABI library builds, loads, exports every entry point declared in
include/gdn.h, and rejects invalid calls on the host before touching a GPU.
(No call here reaches a CUDA API: every case fails validation first.)"""
import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

from gated_deltanet_recurrence_delta_gb300 import build, gdn

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.load_library()


def _declared():
    text = (ROOT / "include" / "gdn.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("gdn_prefill_chunked", "gdn_decode_step", "gdn_verify_with_checkpoints", "gdn_state_copy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def _good_dims(**kw):
    d = dict(B=2, T=1, nk=2, nv=4, dk=32, dv=32, n_slots=2)
    d.update(kw)
    return gdn.make_dims(**d)


def _fake_inputs(base=1 << 20, **over):
    # distinct 16-byte aligned fake device addresses: validation never dereferences them
    names = [f for f, _ in gdn.Inputs._fields_]
    vals = {n: base + 256 * i for i, n in enumerate(names)}
    for n in ("mask", "cu_seqlens", "state_idx"):
        vals[n] = None
    vals.update(over)
    return gdn.Inputs(**vals)


P = 1 << 30  # fake aligned pointer


def _status(fn, *args):
    return fn(*args)


@pytest.mark.parametrize("dims_kw,code", [
    (dict(T=2), "GDN_ERR_SHAPE"),             # decode needs T == 1
    (dict(dk=48, dv=48), "GDN_ERR_SHAPE"),    # unsupported head size
    (dict(dk=32, dv=64), "GDN_ERR_SHAPE"),    # dk != dv
    (dict(nv=3), "GDN_ERR_SHAPE"),            # nv % nk != 0
    (dict(nk=1, nv=16), "GDN_ERR_SHAPE"),     # group > 8
    (dict(n_slots=0), "GDN_ERR_SHAPE"),
    (dict(B=-1), "GDN_ERR_SHAPE"),
])
def test_decode_rejects_bad_dims(lib, dims_kw, code):
    d = _good_dims(**dims_kw)
    st = lib.gdn_decode_step(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, None)
    assert gdn.STATUS[st] == code, gdn.last_error()


def test_decode_rejects_conv_k(lib):
    d = _good_dims(conv_k=3)
    assert gdn.STATUS[lib.gdn_decode_step(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, None)] == "GDN_ERR_SHAPE"


@pytest.mark.parametrize("field", ["q", "k", "v", "z", "a", "b", "A_log", "dt_bias", "conv_w", "norm_w"])
def test_decode_rejects_null_inputs(lib, field):
    d = _good_dims()
    st = lib.gdn_decode_step(ctypes.byref(d), ctypes.byref(_fake_inputs(**{field: None})), P, P, P, None)
    assert gdn.STATUS[st] == "GDN_ERR_ARG"
    assert field in gdn.last_error()


def test_rejects_misaligned_pointer(lib):
    d = _good_dims()
    st = lib.gdn_decode_step(ctypes.byref(d), ctypes.byref(_fake_inputs(q=(1 << 20) + 2)), P, P, P, None)
    assert gdn.STATUS[st] == "GDN_ERR_ARG" and "aligned" in gdn.last_error()
    st = lib.gdn_decode_step(ctypes.byref(d), ctypes.byref(_fake_inputs()), P + 8, P, P, None)
    assert gdn.STATUS[st] == "GDN_ERR_ARG"


def test_null_dims_and_inputs(lib):
    assert gdn.STATUS[lib.gdn_decode_step(None, ctypes.byref(_fake_inputs()), P, P, P, None)] == "GDN_ERR_ARG"
    d = _good_dims()
    assert gdn.STATUS[lib.gdn_decode_step(ctypes.byref(d), None, P, P, P, None)] == "GDN_ERR_ARG"


def test_decode_rejects_cu_seqlens(lib):
    d = _good_dims()
    st = lib.gdn_decode_step(ctypes.byref(d), ctypes.byref(_fake_inputs(cu_seqlens=P)), P, P, P, None)
    assert gdn.STATUS[st] == "GDN_ERR_ARG"


@pytest.mark.parametrize("T", [0, 9])
def test_verify_rejects_T(lib, T):
    d = _good_dims(T=T)
    st = lib.gdn_verify_with_checkpoints(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, P, P, None)
    assert gdn.STATUS[st] == "GDN_ERR_SHAPE"


def test_verify_rejects_null_checkpoints(lib):
    d = _good_dims(T=4)
    st = lib.gdn_verify_with_checkpoints(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, None, P, None)
    assert gdn.STATUS[st] == "GDN_ERR_ARG"


def test_prefill_workspace_rules(lib):
    d = _good_dims(T=100)
    need = lib.gdn_prefill_workspace_size(ctypes.byref(d), 0)
    assert need > 0
    bad = _good_dims(dk=48, dv=48)
    assert lib.gdn_prefill_workspace_size(ctypes.byref(bad), 0) == 0
    st = lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, P, need - 1, None)
    assert gdn.STATUS[st] == "GDN_ERR_WORKSPACE"
    st = lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, None, need, None)
    assert gdn.STATUS[st] == "GDN_ERR_WORKSPACE"
    st = lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, P + 16, need, None)
    assert gdn.STATUS[st] == "GDN_ERR_WORKSPACE"  # not 256-byte aligned


def test_packed_workspace_counts_packed_slots(lib):
    """The size query takes the layout: a packed call (cu_seqlens) of B rows and
    T packed tokens needs T/64 + B + 1 chunk slots, a dense call B * ceil(T/64).
    For the 32 packed varlen rows (lengths U{16..2048} padded to chunk buckets,
    head size 128) the packed size is a small fraction of the dense one."""
    from gated_deltanet_recurrence_delta_gb300 import inputs as I
    _, padded, cu = I.varlen_lengths()
    total = cu[-1]
    d = gdn.make_dims(B=32, T=total, nk=16, nv=32, dk=128, dv=128, n_slots=32)
    dense = gdn.prefill_workspace_size(d, packed=False)
    packed = gdn.prefill_workspace_size(d, packed=True)
    slots_dense, slots_packed = 32 * -(-total // 64), total // 64 + 32 + 1
    assert 0 < packed < dense
    assert packed < 4 * 2**30
    # one slot more per 64 packed tokens; every per-slot image scales with the
    # slot count (the per-row table is tiny)
    d2 = gdn.make_dims(B=32, T=total + 64, nk=16, nv=32, dk=128, dv=128, n_slots=32)
    per_slot = gdn.prefill_workspace_size(d2, packed=True) - packed
    assert abs(per_slot * slots_packed - packed) / packed < 1e-3
    # dense calls also carry the fp16 state image of every (chunk slot, value
    # head) (32 KiB) for the output pass of the few-chain grid
    assert abs((per_slot + 32 * 32768) * slots_dense - dense) / dense < 1e-3
    d3 = gdn.make_dims(B=32, T=total + 128, nk=16, nv=32, dk=128, dv=128, n_slots=32)
    assert abs(gdn.prefill_workspace_size(d3, packed=True) - packed - 2 * per_slot) <= 1024


def test_empty_calls_launch_nothing(lib):
    # B == 0 returns OK before any device work
    d = _good_dims(B=0)
    assert lib.gdn_decode_step(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, None) == 0
    d = _good_dims(B=0, T=3)
    assert lib.gdn_verify_with_checkpoints(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, P, P, None) == 0
    d = _good_dims(T=0)
    assert lib.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(_fake_inputs()), P, P, P, None, 0, None) == 0


def test_state_copy_validation(lib):
    d = _good_dims()
    f = lib.gdn_state_copy
    assert gdn.STATUS[f(ctypes.byref(d), None, None, P, None, P, P, 1, 1, 1, None)] == "GDN_ERR_ARG"
    assert gdn.STATUS[f(ctypes.byref(d), P, P, P, None, P, P, 1, 1, 1, None)] == "GDN_ERR_ARG"  # conv pair
    assert gdn.STATUS[f(ctypes.byref(d), P, None, P, None, P, P, -1, 1, 1, None)] == "GDN_ERR_SHAPE"
    assert gdn.STATUS[f(ctypes.byref(d), P, None, P, None, P, P, 1, 0, 1, None)] == "GDN_ERR_SHAPE"
    assert f(ctypes.byref(d), P, None, P, None, P, P, 0, 1, 1, None) == 0  # nothing to copy


def test_commit_accepted_validation(lib):
    f = lib.gdn_commit_accepted
    d = _good_dims(B=8, T=4, n_slots=3)
    ok = (P, P, P, P, P, P, None, None)  # ckpt_state, ckpt_conv, pools, accept_len, dst_slot, winner, stream
    assert gdn.STATUS[f(ctypes.byref(d), 2, 3, *ok)] == "GDN_ERR_SHAPE"  # 8 rows are not groups of 3
    assert gdn.STATUS[f(ctypes.byref(d), 0, 4, *ok)] == "GDN_ERR_SHAPE"  # no layers
    assert gdn.STATUS[f(ctypes.byref(_good_dims(B=8, T=9)), 2, 4, *ok)] == "GDN_ERR_SHAPE"  # T > 8
    assert gdn.STATUS[f(ctypes.byref(d), 2, 4, P, P, P, P, None, P, None, None)] == "GDN_ERR_ARG"  # accept_len
    assert gdn.STATUS[f(ctypes.byref(d), 2, 4, P, None, P, P, P, P, None, None)] == "GDN_ERR_ARG"  # conv pair
    assert gdn.STATUS[f(ctypes.byref(d), 2, 4, P, P, P, P, P, P, P + 2, None)] == "GDN_ERR_ARG"  # winner alignment
    assert f(ctypes.byref(_good_dims(B=0, T=4)), 2, 4, *ok) == 0  # nothing to commit


def test_decode_mxfp8_validation(lib):
    f = lib.gdn_decode_step_mxfp8
    names = [n for n, _ in gdn.InputsMxfp8._fields_]
    good = {n: (1 << 20) + 256 * i for i, n in enumerate(names)}
    good["mask"] = good["state_idx"] = None
    d = _good_dims()
    inp = gdn.InputsMxfp8(**dict(good, q_scale=None))
    assert gdn.STATUS[f(ctypes.byref(d), ctypes.byref(inp), P, P, P, None)] == "GDN_ERR_ARG"
    inp = gdn.InputsMxfp8(**good)
    assert gdn.STATUS[f(ctypes.byref(_good_dims(T=2)), ctypes.byref(inp), P, P, P, None)] == "GDN_ERR_SHAPE"
    assert gdn.STATUS[f(ctypes.byref(d), ctypes.byref(inp), P, P, None, None)] == "GDN_ERR_ARG"
    assert f(ctypes.byref(_good_dims(B=0)), ctypes.byref(inp), P, P, P, None) == 0


def test_copy_overlapped_validation(lib):
    """Host checks run before anything touches CUDA: a bad count, a NULL list
    or pointer, or an address or size off the 16-byte grid returns an error
    and launches nothing; empty copies are a no-op."""
    f = lib.gdn_copy_overlapped
    C = gdn.Copy

    def call(copies, n=None):
        arr = (C * max(1, len(copies)))(*copies)
        return gdn.STATUS[f(arr, len(copies) if n is None else n, None)]

    good = C(1 << 20, 1 << 21, 4096)
    assert call([good] * 9) == "GDN_ERR_SHAPE"
    assert call([good], n=-1) == "GDN_ERR_SHAPE"
    assert gdn.STATUS[f(None, 1, None)] == "GDN_ERR_ARG"
    assert call([C(None, 1 << 21, 4096)]) == "GDN_ERR_ARG"
    assert call([C(1 << 20, None, 4096)]) == "GDN_ERR_ARG"
    assert call([C((1 << 20) + 8, 1 << 21, 4096)]) == "GDN_ERR_ARG"
    assert call([C(1 << 20, (1 << 21) + 4, 4096)]) == "GDN_ERR_ARG"
    assert call([C(1 << 20, 1 << 21, 4100)]) == "GDN_ERR_ARG"
    assert call([]) == "GDN_OK"
    assert call([C(None, None, 0), C(1 << 20, 1 << 21, 0)]) == "GDN_OK"


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        gdn.load_library(tmp_path / "missing" / "libgdn.so")


def test_commit_source_slot_reading():
    """The commit rule of the speculative verify (generate.py, sparkle:
    commit_tree_row): first path with the longest accept length, its checkpoint
    winner * T + L - 1, nothing (-1) when no token is accepted."""
    from gated_deltanet_recurrence_delta_gb300 import gdn
    assert gdn.commit_source_slot([3, 5, 5, 0], 8) == (1, 1 * 8 + 4)
    assert gdn.commit_source_slot([0, 0, 0], 8) == (0, -1)
    assert gdn.commit_source_slot([8, 2], 8) == (0, 7)
    assert gdn.commit_source_slot([1], 1) == (0, 0)
    assert gdn.commit_source_slot([2, 7, 1, 7, 7], 7) == (1, 7 + 6)
    with pytest.raises(ValueError):
        gdn.commit_source_slot([9], 8)
    with pytest.raises(ValueError):
        gdn.commit_source_slot([], 8)


def test_commit_source_slot_matches_argmax_definition():
    """Against numpy's argmax (first maximum) on random accept lengths: the
    winner and its flat checkpoint index agree on every draw."""
    from gated_deltanet_recurrence_delta_gb300 import gdn
    rng = np.random.default_rng(7)
    for _ in range(500):
        P, T = int(rng.integers(1, 12)), int(rng.integers(1, 10))
        L = rng.integers(0, T + 1, size=P)
        win = int(np.argmax(L))
        assert gdn.commit_source_slot(L, T) == (win, win * T + int(L[win]) - 1 if L[win] > 0 else -1)


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "gdn.h"

int main(void) {
  /* a Qwen3.5-9B-like layer, one 512-token prefill call */
  gdn_dims d;
  memset(&d, 0, sizeof d);
  d.B = 1; d.T = 512; d.nk = 16; d.nv = 32; d.dk = 128; d.dv = 128; d.conv_k = 4; d.n_slots = 1;
  d.scale = 0.08838834764831845f; d.l2_eps = 1e-6f; d.rms_eps = 1e-6f;
  size_t ws = gdn_prefill_workspace_size(&d, 0);
  /* a decode step without inputs: rejected on the host */
  d.T = 1;
  gdn_status st = gdn_decode_step(&d, NULL, NULL, NULL, NULL, NULL);
  const char *msg = gdn_last_error();
  printf("%zu %d %d\n", ws, (int)st, msg != NULL && msg[0] != '\0');
  return 0;
}
"""


def test_plain_c_caller(lib, tmp_path):
    """A C99 program with no CUDA or C++ headers includes gdn.h, links libgdn
    and calls it: the boundary is a plain C ABI. Only host-validated calls are
    made, so no GPU is needed."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc is not installed")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = Path(gdn.LIB_PATH).parent
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", str(ROOT / "include"),
                    str(src), "-o", str(exe), "-L", str(libdir), "-lgdn", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    ws, st, has_msg = int(out[0]), int(out[1]), int(out[2])
    assert ws == gdn.prefill_workspace_size(gdn.make_dims(B=1, T=512, nk=16, nv=32, dk=128, dv=128, n_slots=1))
    assert ws > 0
    assert st == 1 and has_msg == 1  # GDN_ERR_ARG with a message


def test_bench_kernel_source_map_is_complete():
    """Every source the bench maps a kernel to exists (a renamed file would
    break the DRAM-traffic check), and each kernel's code hash computes."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_for_test", ROOT / "bench.py")
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    csrc = ROOT / "gated_deltanet_recurrence_delta_gb300" / "csrc"
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert (csrc / f).is_file(), f"{kernel}: {f} missing"
        assert re.fullmatch(r"[0-9a-f]{16}", bench.csrc_hash(kernel))
