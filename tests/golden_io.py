"""Reader for the hand-worked fixtures in ``tests/golden/`` (input construction only)."""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

from mx_block_scaled_gb300.inputs import FMT_MXFP4, FMT_MXFP8, pack_fp4

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _runs(spec: str, K: int) -> np.ndarray:
    codes = []
    for tok in spec.split():
        code, count = tok.split("*")
        codes += [int(code, 16)] * int(count)
    if len(codes) != K:
        raise ValueError(f"code runs cover {len(codes)} elements, expected {K}")
    return np.array(codes, dtype=np.uint8)


def _value(text: str) -> Fraction:
    text = text.strip()
    if text.startswith("2^"):
        e = int(text[2:])
        return Fraction(2) ** e
    return Fraction(text)


def load_handworked(K: int = 128):
    """Return a list of dicts: name, fmt, A, SA, B, SB (operand arrays), expected (Fraction)."""
    cases = []
    cur = None
    with open(os.path.join(GOLDEN_DIR, "handworked_dot.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            val = val.strip()
            if key == "case":
                cur = {"name": val}
                cases.append(cur)
            elif key == "fmt":
                cur["fmt"] = {"mxfp8": FMT_MXFP8, "mxfp4": FMT_MXFP4}[val]
            elif key in ("a", "b"):
                cur[key] = _runs(val, K)
            elif key in ("sa", "sb"):
                cur[key] = np.array([int(v) for v in val.split()], dtype=np.uint8)
            elif key == "expected":
                cur["expected"] = _value(val)
    out = []
    for c in cases:
        a, b = c["a"][None, :], c["b"][None, :]
        if c["fmt"] == FMT_MXFP4:
            a, b = pack_fp4(a), pack_fp4(b)
        out.append(dict(name=c["name"], fmt=c["fmt"], A=a, B=b,
                        SA=c["sa"][None, :], SB=c["sb"][None, :], expected=c["expected"]))
    return out


def _qvalue(tok: str) -> float:
    t = tok.lower()
    if t in ("nan", "inf", "-inf"):
        return float(t)
    if "x" in t:
        m, e = t.split("x")
        return float(Fraction(m) * Fraction(2) ** int(e))
    return float(Fraction(t)) if t.lstrip("-") != "0" else (-0.0 if t.startswith("-") else 0.0)


def _qruns(spec: str, conv) -> list:
    out = []
    for tok in spec.split():
        val, count = tok.rsplit("*", 1)
        out += [conv(val)] * int(count)
    return out


def load_quantize_handworked():
    """Hand-worked quantisation blocks: list of dicts name, fmt, x (float32 [1, 32]),
    scale (int), codes (uint8 [32], one per element), bf16 (bool)."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN_DIR, "quantize_handworked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            val = val.strip()
            if key == "case":
                cur = {"name": val, "bf16": False}
                cases.append(cur)
            elif key == "fmt":
                cur["fmt"] = {"mxfp8": FMT_MXFP8, "mxfp4": FMT_MXFP4}[val]
            elif key == "x":
                cur["x"] = np.array(_qruns(val, _qvalue), dtype=np.float32)[None, :]
            elif key == "scale":
                cur["scale"] = int(val)
            elif key == "codes":
                cur["codes"] = np.array(_qruns(val, lambda v: int(v, 16)), dtype=np.uint8)
            elif key == "bf16":
                cur["bf16"] = val == "yes"
    for c in cases:
        if c["x"].shape != (1, 32) or c["codes"].shape != (32,):
            raise ValueError(f"case {c['name']}: expected 32 inputs and 32 codes")
    return cases


def _pvalue(tok: str) -> float:
    t = tok.lower()
    if t in ("nan", "inf", "-inf"):
        return float(t)
    if "x" in t:
        m, e = t.split("x")
        return float(Fraction(m) * Fraction(2) ** int(e))
    return float(Fraction(t))


def load_placement_handworked():
    """Hand-worked scale placements: list of dicts k, sa, sb, a (codes), b (codes), pre, post, rn."""
    out = []
    with open(os.path.join(GOLDEN_DIR, "placement_handworked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line.startswith("case:"):
                continue
            head, a, b, vals = [x.strip() for x in line[len("case:"):].split("|")]
            k, sa, sb = (int(v) for v in head.split())
            ac = [int(v, 16) for v in a.split()]
            bc = [int(v, 16) for v in b.split()]
            pre, post, rn = (_pvalue(v) for v in vals.split())
            if len(ac) != k or len(bc) != k:
                raise ValueError(f"placement case {line}: expected {k} codes per operand")
            out.append(dict(k=k, sa=sa, sb=sb, a=ac, b=bc, pre=pre, post=post, rn=rn))
    return out
