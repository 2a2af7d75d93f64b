import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running oracle comparison")


@pytest.fixture(scope="session")
def cuda_lib():
    """The product library on cuda:0; the test fails (not skips) when the CUDA
    extension is missing on a GPU host."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_attention_26_gb300 as pd
    pd.load()  # raises if the library is not built
    return pd


def pytest_terminal_summary(terminalreporter):
    """Achieved parity of every GPU-vs-oracle comparison of the run (passing
    ones included): max-abs, max-rel (over |oracle| >= 1e-3), failing count,
    and the largest share of the tolerance used."""
    mod = sys.modules.get("tests.parity")
    recs = getattr(mod, "RECORDS", None) if mod else None
    if not recs:
        return
    tr = terminalreporter
    tr.section("parity vs oracle (|gpu-oracle| <= 2e-3 + 1e-2|oracle|)")
    worst = {}
    for what, n, mabs, mrel, nbad, use in recs:
        w = worst.get(what)
        if w is None or use > w[4]:
            worst[what] = (n, mabs, mrel, nbad, use)
    tr.write_line(f"{'case':<44} {'elems':>9} {'max_abs':>9} {'max_rel':>9} {'fail':>5} {'tol_used':>8}")
    for what, (n, mabs, mrel, nbad, use) in sorted(worst.items(), key=lambda x: -x[1][4]):
        tr.write_line(f"{what[:44]:<44} {n:>9} {mabs:>9.2e} {mrel:>9.2e} {nbad:>5} {use:>8.3f}")
