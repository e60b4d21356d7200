"""Readers for the hand-derived fixtures under tests/golden/."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [c.strip() for c in line.split("|")]


def pack_cases():
    """(bits, codes uint32[p], expected word) per line of pack_words.txt."""
    out = []
    for bits, codes, word in _rows("pack_words.txt"):
        out.append((int(bits), np.array([int(c) for c in codes.split()], dtype=np.uint32),
                    int(word, 16)))
    return out


def _tile(pattern, n):
    reps = -(-n // len(pattern))
    return (pattern * reps)[:n]


def quant_cases():
    """Quantisation fixtures as dicts with the group's float32 weights built."""
    out = []
    for row in _rows("quant_groups.txt"):
        kind, name, bits, g, sdtype = row[:5]
        bits, g = int(bits), int(g)
        if kind == "built":
            bias, scale, t_pat, q_pat, sbits, bbits = row[5:]
            t = _tile([float(v) for v in t_pat.split()], g)
            q = _tile([int(v) for v in q_pat.split()], g)
            w = np.float32(bias) + np.array(t, dtype=np.float64) * float(scale)
            w32 = w.astype(np.float32)
            assert np.array_equal(w32.astype(np.float64), w), name  # exact by construction
        else:
            w_pat, q_pat, sbits, bbits = row[5:]
            w32 = np.array(_tile([float(v) for v in w_pat.split()], g), dtype=np.float32)
            q = _tile([int(v) for v in q_pat.split()], g)
        out.append(dict(name=name, bits=bits, g=g, sdtype=sdtype, w=w32[None, :],
                        codes=np.array(q, dtype=np.uint32)[None, :],
                        scale_bits=int(sbits, 16), bias_bits=int(bbits, 16)))
    return out
