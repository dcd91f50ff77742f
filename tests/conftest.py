import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name):
    """Parse a tests/golden fixture: '# ...' comments, 'key: values' lines and
    bare rows of numbers.  Returns (dict of key -> list of str, list of rows)."""
    kv, rows = {}, []
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                key, val = line.split(":", 1)
                kv[key.strip()] = val.split()
            else:
                rows.append(line.split())
    return kv, rows


def pytest_terminal_summary(terminalreporter):
    """Report the routing counts the GPU parity tests collected: tokens whose
    top-k boundary gap is below 1e-5 (near_ties), near-tie tokens where the GPU
    chose a different valid set (flips), and clear tokens with two near-equal
    experts in swapped slots (order_swaps)."""
    try:
        from gpu_check import ROUTING_REPORT
    except Exception:
        return
    if not ROUTING_REPORT:
        return
    tot = {"tokens": 0, "near_ties": 0, "flips": 0, "order_swaps": 0}
    terminalreporter.write_sep("-", "routing near-ties (top-k boundary gap < 1e-5)")
    for label, info in ROUTING_REPORT:
        for key in tot:
            tot[key] += info[key]
        if info["near_ties"] or info["flips"] or info["order_swaps"]:
            terminalreporter.write_line(
                f"{label}: tokens={info['tokens']} near_ties={info['near_ties']} "
                f"flips={info['flips']} order_swaps={info['order_swaps']}")
    terminalreporter.write_line(
        f"routing total over {len(ROUTING_REPORT)} checks: tokens={tot['tokens']} "
        f"near_ties={tot['near_ties']} flips={tot['flips']} order_swaps={tot['order_swaps']}")

    try:
        from test_gpu_fp8 import FP8_QUALITY
    except Exception:
        FP8_QUALITY = []
    if FP8_QUALITY:
        terminalreporter.write_sep("-", "FP8 weights: relative L2 of the layer output vs bf16 weights")
        for label, r in FP8_QUALITY:
            terminalreporter.write_line(f"{label}: {r:.3e}")
