import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Print the parity figures of the output comparisons (rows compared, max|gpu - oracle| /
    RMS, and what is left after half an ulp of the output's final rounding), also under -q."""
    helpers = sys.modules.get("helpers")
    recs = [r for r in getattr(helpers, "PARITY_RECORDS", []) if r.get("summary")]
    if not recs:
        return
    terminalreporter.section("output parity: max|gpu-oracle|/RMS raw and after half an ulp of "
                             "the final rounding; worst element in act-rounding sigmas")
    for r in recs:
        z = r.get("max_z")
        terminalreporter.write_line(
            f"{r['what']}: {r['rows']} rows, raw {r['max_err_over_rms']:.4f}, "
            f"minus half ulp {r['max_err_minus_half_ulp_over_rms']:.4f}"
            + ("" if z is None else f", worst {z:.2f} sigma, "
                                    f"{r['over_stated']} elements over 1e-2*RMS + half ulp"))
