"""Pins for the CPU oracle: each check compares the oracle with something other than
itself (the paper's Table 6, closed forms, a library codec, brute force, finite
differences).  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc
from exact_round import code_of_quotient

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ Table 6
def test_table6_format_parameters():
    """NVFP4 (Table 6): blocks of 16, E2M1 elements, E4M3 scales, 4.5 bits/element.
    The oracle's storage per row is K/2 code bytes + K/16 scale bytes."""
    t6 = json.load(open(os.path.join(GOLDEN, "table6_nvfp4_format.json")))
    nv = t6["NVFP4"]
    assert nv["block_size"] == 16
    rng = np.random.default_rng(0)
    for K in (16, 64, 256, 3072):
        q = orc.quantize(rng.standard_normal((3, K)).astype(np.float32))
        assert q.codes.shape == (3, K // 2) and q.scales.shape == (3, K // nv["block_size"])
        bits = 8.0 * (q.codes.shape[1] + q.scales.shape[1]) / K
        assert bits == pytest.approx(nv["bits_per_element"])
    # the MXFP4 column obeys the same storage formula with E8M0 scales per 32
    mx = t6["MXFP4"]
    assert 4 + 8 / mx["block_size"] == pytest.approx(mx["bits_per_element"])
    # element and scale widths: E2M1 = 1+2+1 = 4 bits, E4M3 = 1+4+3 = 8 bits
    assert nv["element_format"] == "E2M1" and nv["block_scale_format"] == "E4M3"


def test_table1_speedups_are_latency_ratios():
    """Internal consistency of the context numbers (Table 1): speedup = BF16/NVFP4."""
    t1 = json.load(open(os.path.join(GOLDEN, "table1_gemm_latency.json")))
    for row in t1["rows"]:
        assert row["bf16_ms"] / row["nvfp4_ms"] == pytest.approx(row["speedup"], abs=0.05)


# ------------------------------------------------------------------ codecs
def _e2m1_closed_form(code):
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return s * mag


def test_e2m1_decode_closed_form_and_roundtrip():
    for c in range(16):
        v = orc.e2m1_decode(c)
        assert v == _e2m1_closed_form(c)
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)
        assert orc.e2m1_encode(v) == c  # exhaustive round trip (incl. -0 -> 0x8)


def _e2m1_brute(v):
    """Nearest E2M1 magnitude by exhaustive distance, ties to the even code."""
    mags = [abs(_e2m1_closed_form(c)) for c in range(8)]
    a = abs(float(v))
    d = [abs(a - m) for m in mags]
    best = min(d)
    cands = [i for i in range(8) if d[i] == best]
    idx = min(cands, key=lambda i: (i % 2, i))  # the even one on a tie
    if a > 6.0:
        idx = 7
    return (8 if math.copysign(1.0, v) < 0 else 0) | idx


def test_e2m1_encode_brute_force_sweep():
    rng = np.random.default_rng(1)
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    vals = list(np.linspace(-8, 8, 4001, dtype=np.float32))
    for m in mids + [0.0, 0.5, 1.0, 6.0, 7.0, 1e-30]:
        for s in (1.0, -1.0):
            x = np.float32(s * m)
            vals += [x, np.nextafter(x, np.float32(100)), np.nextafter(x, np.float32(-100))]
    vals += list((rng.standard_normal(20000) * 3).astype(np.float32))
    vals = np.array(vals, np.float32)
    got = orc.e2m1_encode_array(vals)
    want = np.array([_e2m1_brute(v) for v in vals], np.uint8)
    assert np.array_equal(got, want)
    # the ties named in the design notes
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in ties.items():
        assert orc.e2m1_encode(v) == c
    assert orc.e2m1_encode(-0.1) == 8 and orc.e2m1_encode(-0.0) == 8
    assert orc.e2m1_encode(100.0) == 7 and orc.e2m1_encode(-100.0) == 15


def test_e4m3_decode_matches_torch_codec():
    """All 256 E4M3 bytes against torch's float8_e4m3fn decoder (library routine)."""
    b = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for i in range(256):
        v = orc.e4m3_decode(i)
        if np.isnan(b[i]):
            assert np.isnan(v)
        else:
            assert v == b[i], i
    assert orc.e4m3_decode(0x7E) == 448.0 and orc.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_and_brute_force():
    rng = np.random.default_rng(2)
    finite = np.array([orc.e4m3_decode(c) for c in range(0x7F)], np.float64)  # 0 .. 448
    vals = list(finite)
    mids = (finite[1:] + finite[:-1]) / 2
    for m in mids:
        m32 = np.float32(m)
        vals += [m32, np.nextafter(m32, np.float32(1e9)), np.nextafter(m32, np.float32(0))]
    vals += list(np.exp(rng.uniform(np.log(1e-4), np.log(448.0), 30000)).astype(np.float32))
    vals += [np.float32(1e-9), np.float32(2.0 ** -10), np.float32(447.9)]
    vals = np.array(vals, np.float32)
    got = orc.e4m3_encode_array(vals)
    # library codec (RNE, in range)
    lib = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, lib)
    # brute force over the 127 finite non-negative codes, ties to the even code
    for v, c in zip(vals[::37], got[::37]):
        d = np.abs(finite - float(v))
        best = d.min()
        cands = np.nonzero(d == best)[0]
        idx = cands[0] if len(cands) == 1 else [x for x in cands if x % 2 == 0][0]
        assert c == idx
    # saturation of the finite maximum
    for v in (448.0, 460.0, 480.0, 1e6):
        assert orc.e4m3_encode(v) == 0x7E


# --------------------------------------------------------- per-tensor scale
def test_global_max_block_encodes_448():
    """A block whose amax equals the tensor amax encodes the E4M3 maximum 448, and
    its largest element reconstructs the tensor amax to within FP32 rounding."""
    rng = np.random.default_rng(3)
    for trial in range(50):
        scale = float(np.exp(rng.uniform(-20, 20)))
        x = (rng.standard_normal((8, 64)) * scale).astype(np.float32)
        q = orc.quantize(x)
        a = np.abs(x).max()
        r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert q.scales[r, c // 16] == 0x7E
        xh = orc.dequant(q)
        assert abs(abs(xh[r, c]) - a) <= a * 2.0 ** -21
        assert np.all(q.scales <= 0x7E)


def test_quant_is_nearest_representable():
    """Each scale is the E4M3 value nearest amax_blk/(6g) and each code the E2M1
    value nearest the FP32 quotient RN(x / t), t = RN(e4m3(s) g): the quotient is
    formed from exact rationals here, so an encoder that multiplied by a rounded
    reciprocal instead would fail wherever the two round apart."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((16, 128)) * np.exp(rng.uniform(-3, 3, (16, 1)))).astype(np.float32)
    x[3, 5:21] = 0.0  # a zero block
    q = orc.quantize(x)
    g = q.g
    assert g == np.float32(np.abs(x).max()) / np.float32(2688.0)
    finite = np.array([orc.e4m3_decode(c) for c in range(0x7F)], np.float64)
    codes = orc.unpack_codes(q.codes)
    for r in range(16):
        for b in range(8):
            blk = x[r, b * 16:(b + 1) * 16]
            ratio = np.float32(np.abs(blk).max()) / (np.float32(6.0) * g)
            d = np.abs(finite - float(ratio))
            s_best = np.nonzero(d == d.min())[0]
            s = q.scales[r, b]
            assert s in s_best
            t = np.float32(orc.e4m3_decode(s)) * g
            for i in range(16):
                assert codes[r, b * 16 + i] == code_of_quotient(blk[i], t)


def _near_midpoint_blocks(rng, nblk: int):
    """Blocks of 16 FP32 values, each block's first element fixing the decode step
    t (so that the scale is 448 under g) and the other 15 within a few FP32 steps of
    m t for an E2M1 threshold m: the quotients sit on and around the thresholds."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    g = np.float32(np.exp(rng.uniform(-6, 6)))
    t = np.float32(448.0) * g
    x = np.zeros((nblk, 16), np.float32)
    x[:, 0] = np.float32(2688.0) * g * np.float32(0.999)  # block amax -> scale 448
    for b in range(nblk):
        for i in range(1, 16):
            m = rng.choice(mids)
            v = np.float32(np.float32(m) * t)
            for _ in range(int(rng.integers(-3, 4))):
                v = np.nextafter(v, np.float32(np.inf) if rng.random() < 0.5 else np.float32(0))
            x[b, i] = -v if rng.random() < 0.3 else v
    return x, g


def test_quant_divides_near_thresholds():
    """Quotients on and beside the E2M1 thresholds: the oracle's codes follow the
    exactly rounded quotient x / t, and the same inputs include elements where the
    product with the rounded reciprocal, x * RN(1/t), rounds to another code (so an
    encoder of that order is told apart)."""
    rng = np.random.default_rng(41)
    apart = 0
    for trial in range(40):
        x, g = _near_midpoint_blocks(rng, 8)
        q = orc.quantize(x.reshape(1, -1), g=g)
        codes = orc.unpack_codes(q.codes).reshape(8, 16)
        assert np.all(q.scales == 0x7E)
        t = np.float32(448.0) * g
        rcp = np.float32(1.0) / t
        for b in range(8):
            for i in range(16):
                want = code_of_quotient(x[b, i], t)
                assert codes[b, i] == want
                apart += int(_e2m1_brute(np.float32(x[b, i] * rcp)) != want)
    assert apart > 0


def test_zero_tensor():
    x = np.zeros((4, 32), np.float32)
    x[1, 3] = -0.0
    q = orc.quantize(x)
    assert q.g == 0 and np.all(q.scales == 0)
    assert np.all(orc.dequant(q) == 0)


# ---------------------------------------------------------------- weight pack
def test_weight_pack_transpose_invariant():
    """The backward layout holds exactly the transposed effective weights."""
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((96, 160)) * 0.02).astype(np.float32)
    W[7, 9] = 0.5  # an outlier
    wf, wb = orc.pack_weight(W)
    assert wf.g == wb.g
    df, db = orc.dequant(wf), orc.dequant(wb)
    assert np.array_equal(db, df.T)
    # one scale per 16x16 tile, replicated in both directions
    sf = wf.scales.reshape(6, 16, 10)
    assert np.all(sf == sf[:, :1, :])
    assert np.array_equal(wb.scales.reshape(10, 16, 6)[:, 0, :], sf[:, 0, :].T)
    # the tile holding the tensor amax has scale 448
    assert wf.scales[7, 0] == 0x7E


# --------------------------------------------------------------------- GEMM
def _make_q(rng, R, C, scale_choices=(0x30, 0x38, 0x40)):
    """Random NVFP4 tensor with g = 1 and power-of-two scales (0.5, 1, 2): every
    dequantised value is a multiple of 1/4 and sums of products are exact."""
    codes = rng.integers(0, 256, (R, C // 2), dtype=np.uint8)
    scales = rng.choice(np.array(scale_choices, np.uint8), (R, C // 16))
    return orc.Q(codes, scales, np.float32(1.0), R, C)


def _brute_dequant(q):
    vals = np.zeros((q.rows, q.cols))
    for r in range(q.rows):
        for c in range(q.cols):
            byte = int(q.codes[r, c // 2])
            code = (byte >> 4) if c % 2 else (byte & 15)
            s = int(q.scales[r, c // 16])
            e, m = (s >> 3) & 15, s & 7
            sv = 2.0 ** (e - 7) * (1 + m / 8) if e else 2.0 ** -6 * m / 8
            vals[r, c] = _e2m1_closed_form(code) * sv * float(q.g)
    return vals


def test_tiny_gemm_brute_force_exact():
    rng = np.random.default_rng(6)
    M, K, N, r = 5, 32, 7 * 16 // 16 * 16, 3
    xq = _make_q(rng, M, K)
    wq = _make_q(rng, N, K)
    A = np.zeros((K, r))
    B = np.zeros((r, N))
    y = orc.lora_linear_fwd(xq, wq, A, B, alpha=2.0)
    X, W = _brute_dequant(xq), _brute_dequant(wq)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            want[m, n] = sum(X[m, k] * W[n, k] for k in range(K))
    assert np.array_equal(y, want)


def test_lora_special_cases_exact():
    """B = 0 gives the frozen product alone; W = 0 gives the LoRA branch alone."""
    rng = np.random.default_rng(7)
    M, K, N, r, alpha = 4, 32, 16, 2, 4.0
    xq = _make_q(rng, M, K)
    X = _brute_dequant(xq)
    A = rng.integers(-2, 3, (K, r)).astype(np.float64)
    B = rng.integers(-2, 3, (r, N)).astype(np.float64)
    zero_w = orc.Q(np.zeros((N, K // 2), np.uint8), np.zeros((N, K // 16), np.uint8),
                   np.float32(0.0), N, K)
    y = orc.lora_linear_fwd(xq, zero_w, A, B, alpha)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            want[m, n] = (alpha / r) * sum(sum(X[m, k] * A[k, j] for k in range(K)) * B[j, n]
                                           for j in range(r))
    assert np.array_equal(y, want)
    wq = _make_q(rng, N, K)
    y0 = orc.lora_linear_fwd(xq, wq, A, np.zeros_like(B), alpha)
    assert np.array_equal(y0, X @ _brute_dequant(wq).T)


def test_dgrad_matches_forward_layout_brute_force():
    """dgrad through the backward layout equals sum_n dYhat[m,n] W[n,k] computed by
    brute force from the forward layout (pins the transpose and the LoRA term)."""
    rng = np.random.default_rng(8)
    M, K, N, r, alpha = 3, 32, 48, 2, 2.0
    W = rng.integers(-4, 5, (N, K)).astype(np.float32) * np.float32(0.25)
    wf, wb = orc.pack_weight(W)
    dyq = _make_q(rng, M, N)
    dy = _brute_dequant(dyq)
    A = rng.integers(-2, 3, (K, r)).astype(np.float64)
    B = rng.integers(-2, 3, (r, N)).astype(np.float64)
    prev = rng.integers(-3, 4, (M, K)).astype(np.float64)
    dx = orc.lora_linear_dgrad(dyq, dy, wb, A, B, alpha, dx_prev=prev)
    Wf = _brute_dequant(wf)
    want = np.zeros((M, K))
    for m in range(M):
        for k in range(K):
            base = sum(dy[m, n] * Wf[n, k] for n in range(N))
            lora = sum(sum(dy[m, n] * B[j, n] for n in range(N)) * A[k, j] for j in range(r))
            want[m, k] = base + (alpha / r) * lora + prev[m, k]
    np.testing.assert_allclose(dx, want, rtol=1e-12, atol=1e-9)


def test_fwd_dgrad_adjoint():
    """<fwd(X), D> == <X, dgrad(D)> for the same effective operands (FP64)."""
    rng = np.random.default_rng(9)
    M, K, N, r, alpha = 6, 64, 32, 4, 8.0
    W = (rng.standard_normal((N, K)) * 0.1).astype(np.float32)
    wf, wb = orc.pack_weight(W)
    xq = orc.quantize(rng.standard_normal((M, K)).astype(np.float32))
    dq = orc.quantize(rng.standard_normal((M, N)).astype(np.float32))
    A = rng.standard_normal((K, r))
    B = rng.standard_normal((r, N))
    y = orc.lora_linear_fwd(xq, wf, A, B, alpha)
    dx = orc.lora_linear_dgrad(dq, orc.dequant(dq), wb, A, B, alpha)
    lhs = np.sum(y * orc.dequant(dq))
    rhs = np.sum(orc.dequant(xq) * dx)
    assert lhs == pytest.approx(rhs, rel=1e-12)


def _adapter_grad_is_derivative(grad_fn) -> bool:
    """The forward is linear in A and in B, so for any directions E_A, E_B
    <fwd(A + E_A, B) - fwd(A, B), dY> == <dA, E_A> and likewise for B, exactly up to
    FP64 rounding: the gradients are checked against the forward, not restated."""
    rng = np.random.default_rng(21)
    M, K, N, r, alpha = 9, 64, 48, 5, 10.0
    W = (rng.standard_normal((N, K)) * 0.1).astype(np.float32)
    wf, _ = orc.pack_weight(W)
    xq = orc.quantize(rng.standard_normal((M, K)).astype(np.float32))
    A = rng.standard_normal((K, r))
    B = rng.standard_normal((r, N))
    dy = rng.standard_normal((M, N))
    dA, dB = grad_fn(xq, dy, A, B, alpha)
    if dA.shape != (K, r) or dB.shape != (r, N):
        return False
    loss = lambda A_, B_: float(np.sum(orc.lora_linear_fwd(xq, wf, A_, B_, alpha) * dy))
    base = loss(A, B)
    for _ in range(4):
        EA = rng.standard_normal((K, r))
        EB = rng.standard_normal((r, N))
        if loss(A + EA, B) - base != pytest.approx(float(np.sum(dA * EA)), rel=1e-9, abs=1e-9):
            return False
        if loss(A, B + EB) - base != pytest.approx(float(np.sum(dB * EB)), rel=1e-9, abs=1e-9):
            return False
    return True


def test_adapter_grad_is_the_derivative_of_the_forward():
    assert _adapter_grad_is_derivative(orc.lora_adapter_grad)


def _adapter_grad_planted(kind):
    """The oracle's adapter gradients with one plausible mistake (CPU only)."""
    def grad(xq, dy, A, B, alpha):
        xh = orc.dequant(xq)
        A = np.asarray(A, np.float64)
        B = np.asarray(B, np.float64)
        dy64 = np.asarray(dy, np.float64)
        s = alpha / A.shape[1]
        dA = s * (xh.T @ (dy64 @ B.T))
        dB = s * ((xh @ A).T @ dy64)
        if kind == "scale alpha instead of alpha/r":
            return dA * A.shape[1], dB * A.shape[1]
        if kind == "dA without the input":
            return s * (np.ones_like(xh).T @ (dy64 @ B.T)), dB
        if kind == "dB without the down-projection":
            return dA, s * (np.ones((xh.shape[0], A.shape[1])).T @ dy64)
        if kind == "dB sign":
            return dA, -dB
        raise ValueError(kind)
    return grad


@pytest.mark.parametrize("kind", ["scale alpha instead of alpha/r", "dA without the input",
                                  "dB without the down-projection", "dB sign"])
def test_adapter_grad_pin_catches_planted_mistakes(kind):
    assert not _adapter_grad_is_derivative(_adapter_grad_planted(kind))


def test_adapter_grad_brute_force_and_zero_cases():
    rng = np.random.default_rng(22)
    M, K, N, r, alpha = 3, 16, 16, 2, 4.0
    xq = orc.quantize(rng.integers(-3, 4, (M, K)).astype(np.float32))
    xh = orc.dequant(xq)
    A = rng.integers(-2, 3, (K, r)).astype(np.float64)
    B = rng.integers(-2, 3, (r, N)).astype(np.float64)
    dy = rng.integers(-2, 3, (M, N)).astype(np.float64)
    dA, dB = orc.lora_adapter_grad(xq, dy, A, B, alpha)
    s = alpha / r
    for k in range(K):
        for j in range(r):
            want = s * sum(xh[m, k] * sum(dy[m, n] * B[j, n] for n in range(N)) for m in range(M))
            assert dA[k, j] == pytest.approx(want, abs=1e-12)
    for j in range(r):
        for n in range(N):
            want = s * sum(sum(xh[m, k] * A[k, j] for k in range(K)) * dy[m, n] for m in range(M))
            assert dB[j, n] == pytest.approx(want, abs=1e-12)
    dA0, _ = orc.lora_adapter_grad(xq, dy, A, np.zeros_like(B), alpha)
    _, dB0 = orc.lora_adapter_grad(xq, dy, np.zeros_like(A), B, alpha)
    assert not np.any(dA0) and not np.any(dB0)


# ------------------------------------------------------------- SF swizzle
def test_sf_layout_is_a_bijection_onto_padded_atoms():
    for R, C16 in ((1, 4), (130, 8), (256, 12), (64, 16)):
        Rp, Cp = orc.pad_to(R, 128), orc.pad_to(C16, 4)
        r = np.arange(Rp)[:, None]
        c = np.arange(Cp)[None, :]
        off = orc.sf_offset(r, c, Cp).ravel()
        assert np.array_equal(np.sort(off), np.arange(Rp * Cp))
        s = np.random.default_rng(R).integers(1, 255, (R, C16), dtype=np.uint8)
        flat = orc.swizzle_scales(s)
        assert np.array_equal(orc.unswizzle_scales(flat, R, C16), s)
        assert (flat != 0).sum() == R * C16  # pad bytes are zero


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_rows_closed_form():
    H = 2048
    for c in (1.0, 0.5, 4.0, 2.0 ** -6):
        x = np.full((2, H), c, np.float32)
        gamma = np.ones(H, np.float32)
        rstd, y = orc.rmsnorm_fp32(x, gamma)
        exact = 1.0 / math.sqrt(c * c + float(np.float32(1e-5)))
        assert abs(float(rstd[0]) - exact) <= 2 * np.spacing(np.float32(exact))
        assert np.all(rstd == rstd[0])


def test_rmsnorm_statistic_error_bound_and_output():
    rng = np.random.default_rng(10)
    for H in (16, 48, 512, 3072):
        x = torch.from_numpy(rng.standard_t(3, (7, H)).astype(np.float32)).bfloat16().float().numpy()
        gamma = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
        rstd, y = orc.rmsnorm_fp32(x, gamma)
        ss = (x.astype(np.float64) ** 2).sum(1)
        exact = 1.0 / np.sqrt(ss / H + np.float64(np.float32(1e-5)))
        # FP32 summation of H positive terms: relative error <= H * 2^-24 (loose)
        assert np.all(np.abs(rstd - exact) <= exact * (H + 8) * 2.0 ** -24)
        yref = x.astype(np.float64) * rstd[:, None].astype(np.float64) * gamma[None, :]
        assert np.all(np.abs(y - yref) <= np.abs(yref) * 2.0 ** -22 + 1e-45)


def _rmsnorm_bwd_fd_ok(bwd) -> bool:
    """Whether bwd(y, gamma, rstd, dy) equals central finite differences of an FP64
    RMSNorm forward."""
    rng = np.random.default_rng(11)
    R, H = 3, 32
    x = rng.standard_normal((R, H))
    gamma = 1 + 0.1 * rng.standard_normal(H)
    dy = rng.standard_normal((R, H))
    eps = float(np.float32(1e-5))

    def fwd(xx):
        rs = 1.0 / np.sqrt((xx * xx).mean(1) + eps)
        return xx * rs[:, None] * gamma, rs

    y, rs = fwd(x)
    dx = bwd(y, gamma, rs, dy)
    h = 1e-6
    num = np.zeros_like(x)
    for i in range(R):
        for j in range(H):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            num[i, j] = (np.sum(fwd(xp)[0] * dy) - np.sum(fwd(xm)[0] * dy)) / (2 * h)
    return bool(np.allclose(dx, num, rtol=1e-6, atol=1e-8))


def test_rmsnorm_bwd_finite_differences():
    assert _rmsnorm_bwd_fd_ok(orc.rmsnorm_bwd_from_y)


def _rms_bwd_planted(kind):
    """The oracle's RMSNorm backward with one plausible mistake planted (CPU only)."""
    def bwd(y, gamma, rstd, dy):
        g = np.asarray(gamma, np.float64)[None, :]
        n = np.asarray(y, np.float64) / g
        dn = np.asarray(dy, np.float64) * g
        H = n.shape[1]
        c = (dn * n).sum(axis=1, keepdims=True) / H
        rs = np.asarray(rstd, np.float64)[:, None]
        if kind == "projection term dropped":
            return rs * dn
        if kind == "mean over H - 1":
            return rs * (dn - n * (dn * n).sum(axis=1, keepdims=True) / (H - 1))
        if kind == "gamma not applied to dy":
            return rs * (np.asarray(dy, np.float64) - n * c)
        if kind == "rstd squared":
            return rs * rs * (dn - n * c)
        raise ValueError(kind)
    return bwd


@pytest.mark.parametrize("kind", ["projection term dropped", "mean over H - 1",
                                  "gamma not applied to dy", "rstd squared"])
def test_rmsnorm_bwd_pin_catches_planted_mistakes(kind):
    assert not _rmsnorm_bwd_fd_ok(_rms_bwd_planted(kind))


# -------------------------------------------------------------- exp, SiLU
def test_pexp_accuracy_and_monotonic():
    xs = np.concatenate([np.linspace(-103.9, 88.72, 200001, dtype=np.float32),
                         np.float32([0.0, -0.0, 1.0, -1.0, 1e-8, -1e-8, 0.34657, -0.34657])])
    xs = np.unique(xs)
    ys = orc.pexp(xs)
    ref = np.exp(xs.astype(np.float64))
    normal = ref >= np.finfo(np.float32).tiny
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(ys.astype(np.float64) - ref) / ulp
    assert err[normal].max() <= 2.0
    assert np.all(np.diff(ys.astype(np.float64)) >= 0)
    assert orc.pexp(np.float32([0.0]))[0] == 1.0
    assert np.isinf(orc.pexp(np.float32([89.0]))[0])
    assert orc.pexp(np.float32([-110.0]))[0] == 0.0
    assert np.isfinite(orc.pexp(np.float32([88.7228317]))[0])


def test_silu_mul_special_values():
    g = np.float32([0.0, 50.0, -50.0, 1.0, -200.0, 100.0])
    u = np.float32([3.0, 1.0, 1.0, 1.0, 1.0, 2.0])
    h = orc.silu_mul_fp32(np.concatenate([g, u])[None, :])[0]
    assert h[0] == 0.0
    assert h[1] == 50.0            # silu(x) -> x for large x
    assert abs(h[2]) < 1e-19       # silu(-50) ~ -50 e^-50
    assert abs(h[3] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-7
    assert h[4] == 0.0 and np.signbit(h[4])   # -200 / inf = -0
    assert h[5] == 200.0


def _silu_mul_bwd_fd_ok(bwd) -> bool:
    """Whether bwd(g, u, dh) -> [dgate | dup] equals central finite differences of
    h = g sigmoid(g) u in FP64."""
    rng = np.random.default_rng(12)
    g = rng.standard_normal((2, 16)) * 3
    u = rng.standard_normal((2, 16))
    dh = rng.standard_normal((2, 16))

    def f(gg, uu):
        return np.sum(dh * gg / (1 + np.exp(-gg)) * uu)

    grads = bwd(g, u, dh)
    h = 1e-6
    ng = np.zeros_like(g)
    nu = np.zeros_like(u)
    for i in range(2):
        for j in range(16):
            e = np.zeros_like(g)
            e[i, j] = h
            ng[i, j] = (f(g + e, u) - f(g - e, u)) / (2 * h)
            nu[i, j] = (f(g, u + e) - f(g, u - e)) / (2 * h)
    return bool(np.allclose(grads[:, :16], ng, rtol=1e-6, atol=1e-8) and
                np.allclose(grads[:, 16:], nu, rtol=1e-6, atol=1e-8))


def test_silu_mul_bwd_finite_differences():
    assert _silu_mul_bwd_fd_ok(orc.silu_mul_bwd_from)


def _silu_bwd_planted(kind):
    """The oracle's SiLU-multiply backward with one plausible mistake (CPU only)."""
    def bwd(g, u, dh):
        s = 1.0 / (1.0 + np.exp(-g))
        dgate = dh * u * s * (1.0 + g * (1.0 - s))
        dup = dh * g * s
        if kind == "sigmoid derivative dropped":
            dgate = dh * u * s
        elif kind == "outputs swapped":
            dgate, dup = dup, dgate
        elif kind == "sign of the sigmoid argument":
            sm = 1.0 / (1.0 + np.exp(g))
            dgate = dh * u * sm * (1.0 + g * (1.0 - sm))
            dup = dh * g * sm
        elif kind == "up gradient without gate":
            dup = dh * s
        else:
            raise ValueError(kind)
        return np.concatenate([dgate, dup], axis=1)
    return bwd


@pytest.mark.parametrize("kind", ["sigmoid derivative dropped", "outputs swapped",
                                  "sign of the sigmoid argument", "up gradient without gate"])
def test_silu_mul_bwd_pin_catches_planted_mistakes(kind):
    assert not _silu_mul_bwd_fd_ok(_silu_bwd_planted(kind))


def test_silu_mul_quant_separate_copies():
    """Separate NVFP4 copies of gate and up (Table 7), each with its own scale."""
    rng = np.random.default_rng(13)
    gu = torch.from_numpy(rng.standard_normal((4, 64)).astype(np.float32) * 2).bfloat16().float().numpy()
    gu[:, 32:] *= 10
    hq, gq, uq = orc.silu_mul_quant(gu)
    assert gq.g == orc.global_scale(np.abs(gu[:, :32]).max())
    assert uq.g == orc.global_scale(np.abs(gu[:, 32:]).max())
    assert np.array_equal(orc.dequant(gq), orc.dequant(orc.quantize(gu[:, :32])))


def test_tolerance_helper():
    ref = np.array([1.0, -2.0, 0.0, 3.0])
    ok, worst, _ = orc.check_close(ref * (1 + 7e-3), ref)
    assert ok
    ok, worst, _ = orc.check_close(ref * (1 + 2e-2), ref)
    assert not ok
