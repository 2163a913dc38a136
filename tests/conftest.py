import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library; a GPU test fails loudly when it is missing."""
    from gemm_epilogue_transformer_smem_gb300 import native
    return native.load()


def pytest_terminal_summary(terminalreporter):
    """The unfloored bf16 errors of the comparisons that asked for a report
    (the pass / fail bound is floored at 1% of the tensor RMS; the plain
    relative error and the count of elements above 2e-2 are listed here)."""
    parity = sys.modules.get("parity")
    if parity is None or not (getattr(parity, "REPORTS", None) or getattr(parity, "NOTES", None)):
        return
    tr = terminalreporter
    tr.write_sep("-", "bf16 error vs the fp64 oracle (unfloored relative error; floored bound decides)")
    for name, what, st in parity.REPORTS:
        tr.write_line("%-10s %-10s n=%-9d max|g-r|/|r|=%.3g (|r|=%.2g)  >2e-2: %d  r==0: %d  max err/bound=%.3f" % (
            name, what, st["n"], st["max_rel_unfloored"], st["ref_at_max_rel"],
            st["n_above_2e-2_unfloored"], st["zeros_in_ref"], st["max_err_over_bound"]))
    for note in getattr(parity, "NOTES", []):
        tr.write_line(note)
