"""Shared test helpers: library loading and tolerance checks."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def kosmos():
    import comm_persistent_gemm_gb300 as K
    K.build()
    return K


def header_exports():
    src = open(os.path.join(ROOT, "include", "kosmos.h")).read()
    return sorted(set(re.findall(r"KOSMOS_API\s+[\w\s\*]+?\b(kosmos_\w+)\s*\(", src)))


def rel_err(got, ref):
    """max|got - ref| / max|ref| (the tolerance measure for bf16 outputs)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def bf16_tensor_to_f64(t):
    return t.detach().float().cpu().double().numpy()
