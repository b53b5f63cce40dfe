"""Readers for the text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def hand_products():
    """Parse hand_products.txt into a list of dicts {name, A, B, C, S?}."""
    cases = []
    cur = None
    block = None
    with open(os.path.join(GOLDEN, "hand_products.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                _, name, m, k, n = line.split()
                cur = {"name": name, "dims": (int(m), int(k), int(n))}
                cases.append(cur)
                block = None
            elif line in ("A", "B", "C", "S"):
                block = line
                cur[block] = []
            else:
                cur[block].append([float(v) for v in line.split()])
    for c in cases:
        for key in ("A", "B", "C", "S"):
            if key in c:
                c[key] = np.asarray(c[key], np.float64)
        m, k, n = c["dims"]
        assert c["A"].shape == (m, k) and c["B"].shape == (k, n) and c["C"].shape == (m, n)
    return cases


def page_gflops():
    """Parse page_gflops.txt: rows (N, ms, gflops, ms_decimals)."""
    rows = []
    with open(os.path.join(GOLDEN, "page_gflops.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            n, ms, gf = line.split()
            dec = len(ms.split(".")[1]) if "." in ms else 0
            rows.append((int(n), float(ms), float(gf.replace(",", "")), dec))
    return rows


def update_hand():
    """Parse update_hand.txt into dicts {name, dims, alpha, beta, A, B, C_in, OUT}."""
    cases = []
    cur = None
    block = None
    with open(os.path.join(GOLDEN, "update_hand.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                _, name, m, k, n, alpha, beta = line.split()
                cur = {"name": name, "dims": (int(m), int(k), int(n)),
                       "alpha": float(alpha), "beta": float(beta)}
                cases.append(cur)
                block = None
            elif line in ("A", "B", "C_in", "OUT"):
                block = line
                cur[block] = []
            else:
                cur[block].append([float(v) for v in line.split()])
    for c in cases:
        for key in ("A", "B", "C_in", "OUT"):
            c[key] = np.asarray(c[key], np.float64)
        m, k, n = c["dims"]
        assert c["A"].shape == (m, k) and c["B"].shape == (k, n)
        assert c["C_in"].shape == (m, n) and c["OUT"].shape == (m, n)
    return cases


def tf32_rna():
    """Parse tf32_rna.txt: a list of (input pattern, rounded pattern) as uint32."""
    rows = []
    with open(os.path.join(GOLDEN, "tf32_rna.txt")) as f:
        for raw in f:
            line = raw.split("#")[0].strip()
            if not line:
                continue
            a, b = line.split()
            rows.append((int(a, 16), int(b, 16)))
    return rows
