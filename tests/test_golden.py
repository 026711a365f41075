"""The oracle's MXFP8 element and scale rules against the code points the OCP
specifications fix (tests/golden/e4m3_e8m0_points.txt, each row cited
there)."""
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_e8m0_points.txt")


def _rows(kind):
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line and line[0] == kind:
                out.append(line[1:])
    return out


def _bf16_bits(v):
    u = np.array([v], np.float32).view(np.uint32)[0]
    assert u & 0xFFFF == 0, v  # the fixture's amax values are bf16-exact
    return np.uint16(u >> 16)


def test_e4m3_code_points():
    rows = _rows("e4m3")
    assert len(rows) == 12
    for code_s, value_s in rows:
        code = int(code_s, 16)
        got = oracle.e4m3_decode(code)
        if value_s == "nan":
            assert math.isnan(got), code_s
            continue
        want = float(value_s)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), code_s
        assert oracle.e4m3_encode(want) == code, code_s


def test_e8m0_scale_codes():
    rows = _rows("e8m0")
    assert len(rows) == 6
    for amax_s, code_s, back_s in rows:
        amax = float(amax_s)
        block = np.zeros((1, 32), np.uint16)
        block[0, 5] = _bf16_bits(amax)
        block[0, 6] = _bf16_bits(-amax / 4)
        q, s = oracle.mxfp8_quantize(block)
        code = int(s[0, 0])
        assert code == int(code_s), amax_s
        assert oracle.e4m3_decode(int(q[0, 5])) * 2.0 ** (code - 127) == float(back_s), amax_s
