"""Pins for the oracle's MXFP8 layer (every GEMM operand quantised to MXFP8
along that GEMM's K; the MXFP8 workload of the pages' benchmark set).

* quantisation off: identical to the fp64 layer oracle (pins the plumbing:
  which products are summed, in which order);
* quantisation on: within the MXFP8 error scale of the unquantised layer and
  different from it;
* quantisation axis of one GEMM operand: a huge outlier in one column of the
  down weights flushes the small values sharing its 1x32 blocks to zero only
  when the blocks run along H (the K of the down backward), which changes the
  data gradient by a predictable, large amount;
* the six weight copies equal the quantiser's values along their axes;
* every activation operand, by a flush pin of its own: Xe, Act, dYe, dG/dU
  row blocks along K (forward and data-gradient GEMMs) and the token-axis
  blocks of dYe, Act, Xe, dG, dU (weight-gradient GEMMs). Dropping any one of
  those quantisations from the oracle fails its pin (checked by planting each
  omission in a copy of the oracle);
* locality: a token run alone, or an expert run on exactly its tokens,
  reproduces the whole run's rows; the sampled weight-gradient entries equal
  the whole run's.
"""
import math

import numpy as np
import pytest

import oracle


def _bits(a):
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _layer(N, H, I, E, k, seed):
    rng = np.random.default_rng(seed)
    x = _bits(rng.standard_normal((N, H)))
    wg = _bits(rng.standard_normal((E, I, H)) / math.sqrt(H))
    wu = _bits(rng.standard_normal((E, I, H)) / math.sqrt(H))
    wd = _bits(rng.standard_normal((E, H, I)) / math.sqrt(H))
    dy = _bits(rng.standard_normal((N, H)))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    w = rng.random((N, k)) + 0.1
    w /= w.sum(1, keepdims=True)
    return x, wg, wu, wd, ids, w, dy


def test_without_quantisation_equals_the_layer_oracle():
    x, wg, wu, wd, ids, w, dy = _layer(40, 64, 96, 5, 2, 1)
    r = oracle.layer_mxfp8(x, wg, wu, wd, ids, w, dy, quantize=False)
    yb = oracle.forward_bf16(x, wg, wu, wd, ids, w)
    rb = oracle.backward_bf16(x, wg, wu, wd, ids, w, dy)
    np.testing.assert_array_equal(r["y"], yb)
    for key in ("dx", "dwg", "dwu", "dwd", "dw"):
        np.testing.assert_array_equal(r[key], rb[key])


def test_quantised_layer_stays_within_the_mxfp8_error_scale():
    x, wg, wu, wd, ids, w, dy = _layer(64, 64, 96, 4, 2, 2)
    r = oracle.layer_mxfp8(x, wg, wu, wd, ids, w, dy, quantize=True)
    ref = oracle.layer_mxfp8(x, wg, wu, wd, ids, w, dy, quantize=False)
    for key in ("y", "dx", "dwg", "dwu", "dwd", "dw"):
        err = np.max(np.abs(r[key] - ref[key])) / np.max(np.abs(ref[key]))
        # E4M3 keeps 3 mantissa bits (relative rounding <= 2^-4 per operand);
        # a few quantised factors per output stay well inside 0.25
        assert 1e-4 < err < 0.25, (key, err)


def test_down_backward_quantises_wd_along_h():
    """dx depends on Wd only through dA = Wd^T dYe, whose K is H. An outlier
    2^20 times larger than the rest in Wd[0][0][i] shares its H-blocks
    (h = 0..31, fixed i) with 31 small values that then flush to zero, so
    dA[i] loses their contribution for every i of the outlier row. Putting the
    outliers in a whole row h = 0 makes the flush cover every i."""
    N, H, I, E, k = 3, 64, 64, 1, 1
    x, wg, wu, wd, ids, w, dy = _layer(N, H, I, E, k, 3)
    wd_f = oracle.bf16_bits_to_f64(wd)
    wd_f[0, 0, :] = 2.0 ** 20
    wd_out = _bits(wd_f)
    base = oracle.layer_mxfp8(x, wg, wu, wd_out, ids, w, dy, quantize=True)
    # Same weights but rows h = 1..31 of Wd zeroed: if Wd is quantised along
    # H those rows are flushed anyway, so dx must not change at all.
    wd_z = wd_f.copy()
    wd_z[0, 1:32, :] = 0.0
    flushed = oracle.layer_mxfp8(x, wg, wu, _bits(wd_z), ids, w, dy, quantize=True)
    np.testing.assert_array_equal(base["dx"], flushed["dx"])
    # ... while without quantisation zeroing those rows does change dx
    a = oracle.layer_mxfp8(x, wg, wu, wd_out, ids, w, dy, quantize=False)
    b = oracle.layer_mxfp8(x, wg, wu, _bits(wd_z), ids, w, dy, quantize=False)
    assert np.max(np.abs(a["dx"] - b["dx"])) > 0


def test_weight_copies_are_the_quantiser_s_values_and_the_two_halves_compose():
    """The prepared weight copies hold the decoded MXFP8 values of each row
    (blocks along the stored axis) or of each column (blocks across it), and
    weights-then-layer gives exactly the one-call layer."""
    x, wg, wu, wd, ids, w, dy = _layer(24, 64, 96, 3, 2, 3)
    pw = oracle.mxfp8_weights(wg, wu, wd)

    def dequant(bits2d):
        q, s = oracle.mxfp8_quantize(bits2d)
        vals = np.array([oracle.e4m3_decode(c) for c in range(256)])
        scale = np.exp2(s.astype(np.float64) - 127.0)
        return vals[q] * np.repeat(scale, 32, axis=1)

    e = 1
    np.testing.assert_array_equal(pw["wg_h"][e], dequant(wg[e]))
    np.testing.assert_array_equal(pw["wd_i"][e], dequant(wd[e]))
    np.testing.assert_array_equal(pw["wu_i"][e], dequant(np.ascontiguousarray(wu[e].T)).T)
    np.testing.assert_array_equal(pw["wd_h"][e], dequant(np.ascontiguousarray(wd[e].T)).T)
    r1 = oracle.layer_mxfp8(x, wg, wu, wd, ids, w, dy)
    r2 = oracle.layer_mxfp8_prepared(x, pw, ids, w, dy)
    for key in r1:
        np.testing.assert_array_equal(r1[key], r2[key])


def test_token_rows_and_expert_segments_are_local():
    """What the full-size sampled MXFP8 parity test relies on. Every forward
    and dX-path operand is quantised along K one row at a time, so a token
    run alone against its own k experts gives its y, dx and d(routing
    weights) exactly. An expert's weight-gradient operands are quantised in
    32-token blocks from the start of its segment (tokens ascending), so that
    expert run alone on exactly its tokens (k = 1) gives its dW exactly --
    and the same tokens in another order do not (the blocks regroup)."""
    N, H, I, E, k = 80, 64, 96, 3, 2  # ~53 tokens per expert: a ragged 32-token block
    x, wg, wu, wd, ids, w, dy = _layer(N, H, I, E, k, 5)
    full = oracle.layer_mxfp8(x, wg, wu, wd, ids, w, dy)
    own = np.arange(k, dtype=np.int32)[None]
    for t in (0, 41, N - 1):
        ex = ids[t]
        r = oracle.layer_mxfp8(x[t:t + 1], wg[ex], wu[ex], wd[ex], own, w[t:t + 1], dy[t:t + 1])
        for key in ("y", "dx", "dw"):
            np.testing.assert_array_equal(r[key][0], full[key][t])
    for e in range(E):
        hit = ids == e
        toks = np.flatnonzero(hit.any(axis=1))
        assert len(toks) % 32 != 0
        one = np.zeros((len(toks), 1), np.int32)
        r = oracle.layer_mxfp8(x[toks], wg[e:e + 1], wu[e:e + 1], wd[e:e + 1], one,
                               w[hit][:, None], dy[toks])
        for key in ("dwg", "dwu", "dwd"):
            np.testing.assert_array_equal(r[key][0], full[key][e])
        rev = toks[::-1]
        r = oracle.layer_mxfp8(x[rev], wg[e:e + 1], wu[e:e + 1], wd[e:e + 1], one,
                               w[hit][::-1, None], dy[rev])
        assert not np.array_equal(r["dwd"][0], full["dwd"][e])


@pytest.mark.parametrize("quantize", [True, False])
def test_sampled_expert_wgrad_equals_the_layer_entries(quantize):
    """expert_wgrad_mxfp8 (sampled entries, any expert size) against the
    whole-layer oracle: equal entries, bit for bit, on ragged experts and on
    lists that repeat, reorder and reach the last row and column."""
    N, H, I, E, k = 90, 64, 96, 3, 2
    x, wg, wu, wd, ids, w, dy = _layer(N, H, I, E, k, 8)
    full = oracle.layer_mxfp8(x, wg, wu, wd, ids, w, dy, quantize=quantize)
    il = np.array([95, 0, 31, 32, 7, 7], np.int32)
    hl = np.array([63, 1, 32, 0, 40], np.int32)
    for e in range(E):
        r = oracle.expert_wgrad_mxfp8(x, wg, wu, wd, ids, w, dy, e, il, hl, quantize=quantize)
        np.testing.assert_array_equal(r["dwg"], full["dwg"][e][np.ix_(il, hl)])
        np.testing.assert_array_equal(r["dwu"], full["dwu"][e][np.ix_(il, hl)])
        np.testing.assert_array_equal(r["dwd"], full["dwd"][e][np.ix_(hl, il)])


def test_sampled_expert_wgrad_rejects_bad_lists():
    x, wg, wu, wd, ids, w, dy = _layer(8, 64, 96, 3, 2, 1)
    with pytest.raises(oracle.OracleError):
        oracle.expert_wgrad_mxfp8(x, wg, wu, wd, ids, w, dy, 0, [96], [0])
    with pytest.raises(oracle.OracleError):
        oracle.expert_wgrad_mxfp8(x, wg, wu, wd, ids, w, dy, 3, [0], [0])


# Flush pins for the activation operands. Each plants an outlier 2^40 times
# the typical magnitude at position 0 of a 32-value block of one operand; with
# that operand quantised along the block's axis the other 31 values of the
# block round to zero (E4M3 keeps values down to 2^-17 of the block maximum),
# so zeroing their sources leaves the watched output bit-identical -- and
# without quantisation the same edit changes it. Zeroing in one place only
# (the operand's own inputs) keeps every other operand's blocks unchanged.
BIG = 2.0 ** 40


def _flush_pair(make, watch):
    x, wg, wu, wd, ids, w, dy = _layer(3, 64, 64, 1, 1, 11)
    args_a, args_b = make(x, wg, wu, wd, dy)
    for quantize, same in ((True, True), (False, False)):
        ra = oracle.layer_mxfp8(*args_a[:4], ids, w, args_a[4], quantize=quantize)
        rb = oracle.layer_mxfp8(*args_b[:4], ids, w, args_b[4], quantize=quantize)
        assert np.array_equal(watch(ra), watch(rb)) == same, quantize


def test_xe_rows_are_quantised_along_h():
    """y[t] sees x[t] only through Xe's rows, 32-blocks along H. Column h = 0
    of Wg and Wu is zero, so the outlier x[t, 0] sets its block's scale but
    adds nothing to G and U (else it would swamp the neighbours' share below
    the bf16 rounding of Act and hide a missing quantisation)."""
    def make(x, wg, wu, wd, dy):
        wgf, wuf = oracle.bf16_bits_to_f64(wg), oracle.bf16_bits_to_f64(wu)
        wgf[:, :, 0] = 0.0
        wuf[:, :, 0] = 0.0
        xf = oracle.bf16_bits_to_f64(x)
        xf[1, 0] = BIG
        xz = xf.copy()
        xz[1, 1:32] = 0.0
        wg0, wu0 = _bits(wgf), _bits(wuf)
        return (_bits(xf), wg0, wu0, wd, dy), (_bits(xz), wg0, wu0, wd, dy)
    _flush_pair(make, lambda r: r["y"][1])


def test_act_rows_are_quantised_along_i():
    """Wu[0][0][:] scaled by 2^40 makes Act[:, 0] the outlier of block
    i = 0..31; zeroing Wg and Wu rows 1..31 (their own row blocks along H are
    independent) makes Act[:, 1:32] exactly 0 instead of flushed."""
    def make(x, wg, wu, wd, dy):
        wuf = oracle.bf16_bits_to_f64(wu)
        wuf[0, 0, :] *= BIG
        wgz, wuz = oracle.bf16_bits_to_f64(wg), wuf.copy()
        wgz[0, 1:32, :] = 0.0
        wuz[0, 1:32, :] = 0.0
        return (x, wg, _bits(wuf), wd, dy), (x, _bits(wgz), _bits(wuz), wd, dy)
    _flush_pair(make, lambda r: r["y"])


def test_dye_rows_are_quantised_along_h():
    """dx[t] sees dY[t] only through dYe's rows, 32-blocks along H (dw, the
    routing-weight gradient, reads dY unquantised and is not watched). Row
    h = 0 of Wd is zero, so the outlier dY[t, 0] sets its block's scale but
    adds nothing to dAct."""
    def make(x, wg, wu, wd, dy):
        wdf = oracle.bf16_bits_to_f64(wd)
        wdf[0, 0, :] = 0.0
        wd0 = _bits(wdf)
        df = oracle.bf16_bits_to_f64(dy)
        df[2, 0] = BIG
        dz = df.copy()
        dz[2, 1:32] = 0.0
        return (x, wg, wu, wd0, _bits(df)), (x, wg, wu, wd0, _bits(dz))
    _flush_pair(make, lambda r: r["dx"][2])


def test_dg_du_rows_are_quantised_along_i():
    """Wd[0][:][0] scaled by 2^40 makes dAct[:, 0], hence dG[:, 0] and
    dU[:, 0], the outliers of block i = 0..31; zeroing Wd columns 1..31 makes
    dAct, dG, dU exactly 0 there instead of flushed. The forward's Wd row
    blocks along I already flush those columns, and Wd's column blocks along H
    are per column, so nothing else changes."""
    def make(x, wg, wu, wd, dy):
        wdf = oracle.bf16_bits_to_f64(wd)
        wdf[0, :, 0] *= BIG
        wdz = wdf.copy()
        wdz[0, :, 1:32] = 0.0
        return (x, wg, wu, _bits(wdf), dy), (x, wg, wu, _bits(wdz), dy)
    _flush_pair(make, lambda r: r["dx"])


# The same flush pins for the weight-gradient operands, whose 32-value blocks
# run along the token axis of an expert's segment (E = 1, k = 1, 40 tokens:
# tokens 0..31 form the first block). The outlier sits at token 0; zeroing
# the sources of tokens 1..31 leaves the watched gradient bit-identical only
# if that operand is quantised along tokens. Sums of the weight gradients are
# fp64 with no rounding, so an unquantised operand's O(1) terms beside the
# 2^40-scale one would show.
def _wgrad_pair(make, watch):
    x, wg, wu, wd, ids, w, dy = _layer(40, 64, 64, 1, 1, 12)
    args_a, args_b = make(x, wg, wu, wd, dy)
    for quantize, same in ((True, True), (False, False)):
        ra = oracle.layer_mxfp8(*args_a[:4], ids, w, args_a[4], quantize=quantize)
        rb = oracle.layer_mxfp8(*args_b[:4], ids, w, args_b[4], quantize=quantize)
        assert np.array_equal(watch(ra), watch(rb)) == same, quantize


def test_dye_columns_are_quantised_along_tokens():
    """dWd[h0, :] = sum over tokens of dYe[:, h0] * Act: dY[0, h0] is the
    outlier of dYe's first token block in column h0. Zeroing dY[1:32, h0]
    changes only dYe (and, through its row blocks, dAct, which dWd does not
    read)."""
    h0 = 5

    def make(x, wg, wu, wd, dy):
        df = oracle.bf16_bits_to_f64(dy)
        df[0, h0] = BIG
        dz = df.copy()
        dz[1:32, h0] = 0.0
        return (x, wg, wu, wd, _bits(df)), (x, wg, wu, wd, _bits(dz))
    _wgrad_pair(make, lambda r: r["dwd"][0, h0])


def test_act_columns_are_quantised_along_tokens():
    """x[0] scaled by 2^12 makes Act[0, i0] (i0 with G and U well away from 0
    for token 0) the outlier of Act's first token block in column i0; zeroing
    x rows 1..31 makes their Act exactly 0. dYe is untouched, so dWd[:, i0]
    can change only through Act's column blocks."""
    def make(x, wg, wu, wd, dy):
        xf = oracle.bf16_bits_to_f64(x)
        g = oracle.bf16_bits_to_f64(wg)[0] @ xf[0]
        u = oracle.bf16_bits_to_f64(wu)[0] @ xf[0]
        i0 = int(np.argmax(np.where(g > 0, g * np.abs(u), -np.inf)))
        make.i0 = i0
        xf[0] *= 2.0 ** 12
        xz = xf.copy()
        xz[1:32] = 0.0
        return (_bits(xf), wg, wu, wd, dy), (_bits(xz), wg, wu, wd, dy)
    _wgrad_pair(make, lambda r: r["dwd"][0][:, make.i0])


def test_xe_columns_are_quantised_along_tokens():
    """dWg[:, h0], dWu[:, h0] read x[:, h0] through Xe's token blocks.
    Column h0 of Wg and Wu is zero, so x[:, h0] changes no G or U; the values
    x[1:32, h0] are made small so they never set their row block's scale."""
    h0 = 7

    def make(x, wg, wu, wd, dy):
        wgf, wuf = oracle.bf16_bits_to_f64(wg), oracle.bf16_bits_to_f64(wu)
        wgf[:, :, h0] = 0.0
        wuf[:, :, h0] = 0.0
        xf = oracle.bf16_bits_to_f64(x)
        xf[0, h0] = BIG
        xf[1:32, h0] = 2.0 ** -6
        xz = xf.copy()
        xz[1:32, h0] = 0.0
        wg0, wu0 = _bits(wgf), _bits(wuf)
        return (_bits(xf), wg0, wu0, wd, dy), (_bits(xz), wg0, wu0, wd, dy)
    _wgrad_pair(make, lambda r: np.concatenate([r["dwg"][0][:, h0], r["dwu"][0][:, h0]]))


def test_dg_du_columns_are_quantised_along_tokens():
    """dY[0] scaled by 2^40 scales dYe, dAct, dG and dU of token 0 by 2^40
    (a power of two passes through every rounding unchanged), making token 0
    the outlier of every dG and dU column's first token block; zeroing dY
    rows 1..31 makes their dG and dU exactly 0. x is untouched, so dWg and dWu
    can change only through dG's and dU's column blocks."""
    def make(x, wg, wu, wd, dy):
        df = oracle.bf16_bits_to_f64(dy)
        df[0] *= BIG
        dz = df.copy()
        dz[1:32] = 0.0
        return (x, wg, wu, wd, _bits(df)), (x, wg, wu, wd, _bits(dz))
    _wgrad_pair(make, lambda r: np.concatenate([r["dwg"].ravel(), r["dwu"].ravel()]))


def test_trace_without_the_diagnostic_equals_the_layer_and_exposes_dg_du():
    """The error-accounting entry (layer_mxfp8_trace): with gu_bf16 off every
    output equals layer_mxfp8 bit for bit; the dG/dU rows it exposes are the
    operands of the gate/up data gradient (dx recomputed from them and the
    transposed weight copies matches), and each is an MXFP8 number along I
    (a fixed point of the quantiser)."""
    x, wg, wu, wd, ids, w, dy = _layer(24, 64, 96, 5, 2, 7)
    prep = oracle.mxfp8_weights(wg, wu, wd)
    r = oracle.layer_mxfp8(x, wg, wu, wd, ids, w, dy, quantize=True)
    t = oracle.layer_mxfp8_trace(x, prep, ids, w, dy, gu_bf16=False)
    for key in ("y", "dx", "dwg", "dwu", "dwd", "dw"):
        np.testing.assert_array_equal(t[key], r[key], err_msg=key)
    N, k = ids.shape
    dx = np.zeros_like(r["dx"])
    for a in range(N * k):
        e = ids.reshape(-1)[a]
        dx[a // k] += prep["wg_i"][e].T @ t["dg_rows"][a] + prep["wu_i"][e].T @ t["du_rows"][a]
    np.testing.assert_allclose(dx, r["dx"], rtol=0, atol=1e-12 * np.max(np.abs(r["dx"])))
    for rows in (t["dg_rows"], t["du_rows"]):
        q = _qdq_rows(rows)
        np.testing.assert_array_equal(q, rows)


def _qdq_rows(v):
    """Quantise-dequantise rows of exact bf16 values along the row (blocks of
    32) with the oracle's element and scale rules."""
    q, s = oracle.mxfp8_quantize(_bits(v.astype(np.float32)))
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    return table[q] * np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)


def test_trace_bf16_gu_changes_only_the_swiglu_backward_outputs():
    """gu_bf16 rounds G and U before the SwiGLU backward: y, dWd and d(routing
    weights) do not depend on it; dx, dWg and dWu move by a small amount."""
    x, wg, wu, wd, ids, w, dy = _layer(24, 64, 96, 5, 2, 8)
    prep = oracle.mxfp8_weights(wg, wu, wd)
    a = oracle.layer_mxfp8_trace(x, prep, ids, w, dy, gu_bf16=False)
    b = oracle.layer_mxfp8_trace(x, prep, ids, w, dy, gu_bf16=True)
    for key in ("y", "dwd", "dw"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    for key in ("dx", "dwg", "dwu"):
        d = np.max(np.abs(a[key] - b[key])) / np.max(np.abs(a[key]))
        assert 0 < d < 0.1, (key, d)
