import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """The parity margins the GPU tests measured: per test the worst bf16 output
    error beyond the output's own rounding (bar 2e-2), the raw max-abs, and the
    worst relative Frobenius error of a final state (bar 1e-3); the worst of
    each last. With GDN_PARITY_LOG set they are also written there as JSON."""
    gc = sys.modules.get("tests.gpu_cases")
    margins = getattr(gc, "MARGINS", None) if gc else None
    if not margins:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins (out: beyond half a bf16 ulp, bar 2e-2 | raw max-abs | state rel-Fro, bar 1e-3)")
    for tid in sorted(margins):
        m = margins[tid]
        name = tid.split("::", 1)[-1]
        extra = "".join(f" {k} {v:.2e}" for k, v in sorted(m.items())
                        if k not in ("out_beyond_half_ulp", "out_raw_max_abs", "state_rel_fro"))
        tr.write_line(f"{name[:70]:70s} out {m.get('out_beyond_half_ulp', float('nan')):9.2e} "
                      f"raw {m.get('out_raw_max_abs', float('nan')):9.2e} "
                      f"state {m.get('state_rel_fro', float('nan')):9.2e}{extra}")
    for kind, bar in (("out_beyond_half_ulp", 2e-2), ("out_raw_max_abs", None), ("state_rel_fro", 1e-3)):
        vals = [(m[kind], t) for t, m in margins.items() if kind in m]
        if vals:
            v, t = max(vals)
            tr.write_line(f"worst {kind}: {v:.3e}" + (f" (bar {bar:g})" if bar else "") + f" in {t.split('::', 1)[-1]}")
    path = os.environ.get("GDN_PARITY_LOG")
    if path:
        import json
        Path(path).parent.mkdir(parents=True, exist_ok=True)
        Path(path).write_text(json.dumps(margins, indent=1, sort_keys=True))
