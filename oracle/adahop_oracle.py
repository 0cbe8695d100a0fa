"""AdaHOP oracle: a plain, slow CPU restatement of the outlier-pattern-aware MXFP4 linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
use it.  It shares no code with the CUDA library; the only thing both sides use is the seeded
input generator in ``synthetic/``.

What it follows (AdaHOP: Fast and Accurate Low-Precision Training via Outlier-Pattern-Aware
Rotation, Kim, Khodamoradi, Denolf, Park, arXiv 2604.02525):

* abstract: three outlier patterns (Row-wise, Column-wise, None); the Inner Hadamard
  Transform (IHT) when mixing along the inner dimension suppresses the outliers, otherwise
  Outlier Extraction (OE) of dominant rows/columns into a high-precision (BF16) path;
* Fig. 2: a Right Hadamard suppresses column-wise outliers, a Left one leaves them intact;
* Fig. 5: each linear runs three matmuls (Fwd, dX, dW); each picks IHT, OE-Left, OE-Right or
  BF16 from its operand pattern pair;
* Fig. 9 and the appendix implementation notes: FOID (variance of the first 64 elements of
  every row or column, top-k lines become outliers, their entries are zeroed in the residual),
  IHT + quantisation (1D FWHT with block size 32 on the residual, then MXFP4 with 1D scaling),
  a GEMM over the MXFP4 residual plus the BF16 outliers, and an in-place scatter-add of the
  outlier product;
* MXFP4 itself (E2M1 elements, one E8M0 scale per 32 elements) is the OCP Microscaling
  Formats v1.0 definition, which the pages name but do not restate.

Readings taken where the pages are silent, numbered R1-R11:

R1  calibration: mean-square per row and per column, ratio of the max to the lower median,
    threshold tau = 8; Column-wise if the column ratio wins, else Row-wise.
R2, R3  pattern pair -> strategy: CN, NN -> IHT; RC, RN -> OE-Left; NC -> OE-Right; every other
    pair -> BF16.  OE-Left takes rows of the Row-wise operand (A-source if none/both),
    OE-Right takes columns of the Column-wise operand (B-source if none/both).
R4  FOID score: population variance of the first 64 elements in float32, summed by a fixed
    pairwise tree (i + 32, then + 16, ... + 1), no fused multiply-add; ties to the lower index;
    indices returned ascending.
R5  Hadamard: Sylvester order, orthonormal (times the float32 nearest 1/sqrt(32)), not
    randomised; butterflies with stride 1, 2, 4, 8, 16 in float32.
R6-R8  MX scale: E8M0 byte = clamp(floor(log2 amax) - 2 + 127, 0, 254); an all-zero block has
    byte 0 and codes 0; elements round to the nearest E2M1 value, ties to the even code,
    saturating at 6; the sign bit is the element's sign bit; the even element sits in the low
    nibble.  The scale axis is the GEMM's inner dimension.
R9, R10  inner OE zeroes only the extracting operand; the partner keeps its lines.  The residual of
    every OE strategy also gets the IHT before quantisation.
R11  outer OE: the residual's extracted rows (columns) of C are exactly zero, so the scatter-add
    result is the outlier product rounded once to the output type.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

# --------------------------------------------------------------------------------------------
# Enumerations (the pages' vocabulary)
# --------------------------------------------------------------------------------------------
PAT_NONE, PAT_ROW, PAT_COL = 0, 1, 2
PATTERN_LETTER = {PAT_NONE: "N", PAT_ROW: "R", PAT_COL: "C"}

IHT, OE_LEFT, OE_RIGHT, BF16, MXFP4_PLAIN = 0, 1, 2, 3, 4
STRATEGY_NAME = {IHT: "IHT", OE_LEFT: "OE-Left", OE_RIGHT: "OE-Right", BF16: "BF16",
                 MXFP4_PLAIN: "MXFP4"}

GEMMS = ("fwd", "dgrad", "wgrad")

# E2M1 magnitudes, indexed by the 3-bit code (exponent bits, mantissa bit).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
MX_BLOCK = 32
FOID_PROBE = 64
DEFAULT_TAU = 8.0
DEFAULT_RANK = 64


# --------------------------------------------------------------------------------------------
# bf16 helpers (plain bit manipulation)
# --------------------------------------------------------------------------------------------
def bf16_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); finite inputs only."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------------------------
# Hadamard (reading R5)
# --------------------------------------------------------------------------------------------
def _nearest_f32_inv_sqrt32() -> np.float32:
    """The float32 value nearest 1/sqrt(32), confirmed with exact rational arithmetic.

    x = 1/sqrt(32) is irrational, so c is the nearest float32 iff x lies strictly between the
    midpoints of c with its two neighbours, i.e. m_lo^2 < 1/32 < m_hi^2.
    """
    target = Fraction(1, 32)
    c0 = np.float32(1.0 / np.sqrt(32.0))
    for c in (c0, np.nextafter(c0, np.float32(0)), np.nextafter(c0, np.float32(1))):
        f = Fraction(float(c))
        m_lo = (Fraction(float(np.nextafter(c, np.float32(0)))) + f) / 2
        m_hi = (Fraction(float(np.nextafter(c, np.float32(1)))) + f) / 2
        if m_lo * m_lo < target < m_hi * m_hi:
            return np.float32(c)
    raise AssertionError("no float32 brackets 1/sqrt(32)")


INV_SQRT32_F32 = _nearest_f32_inv_sqrt32()


def hadamard_matrix(n: int = MX_BLOCK, normalized: bool = True) -> np.ndarray:
    """Sylvester Hadamard H_n (natural order): H_1 = [1], H_2k = [[H, H], [H, -H]]."""
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    if h.shape[0] != n:
        raise ValueError("n must be a power of two")
    return h / np.sqrt(n) if normalized else h


def fwht32_f32(z) -> np.ndarray:
    """Block-32 fast Walsh-Hadamard transform along the last axis, in float32.

    Butterflies with stride h = 1, 2, 4, 8, 16: (a, b) -> (a + b, a - b), each rounded to
    float32, then one multiplication by the float32 constant nearest 1/sqrt(32).
    (AdaHOP appendix implementation notes, IHT and Quantization: 1D FWHT, block size 32.)
    """
    y = np.array(z, dtype=np.float32, copy=True)
    shape = y.shape
    if shape[-1] % MX_BLOCK:
        raise ValueError("last axis must be a multiple of 32")
    y = y.reshape(-1, MX_BLOCK)
    h = 1
    while h < MX_BLOCK:
        v = y.reshape(-1, MX_BLOCK // (2 * h), 2, h)
        a = v[:, :, 0, :].copy()
        b = v[:, :, 1, :].copy()
        v[:, :, 0, :] = a + b
        v[:, :, 1, :] = a - b
        h *= 2
    y = y * INV_SQRT32_F32
    return y.reshape(shape)


# --------------------------------------------------------------------------------------------
# MXFP4 (readings R6-R8; OCP MX v1.0 element and scale formats)
# --------------------------------------------------------------------------------------------
def mx_scale_bytes(amax) -> np.ndarray:
    """E8M0 scale byte per block: clamp(floor(log2 amax) - 2 + 127, 0, 254); 0 for amax = 0.

    floor(log2 amax) is read off frexp, which is exact for every float32 (subnormals too).
    """
    a = np.asarray(amax, dtype=np.float32).astype(np.float64)
    _, e = np.frexp(a)            # a = m * 2^e, m in [0.5, 1)  =>  floor(log2 a) = e - 1
    e = e.astype(np.int64) - 1
    byte = np.clip(e - 2 + 127, 0, 254)
    return np.where(a > 0, byte, 0).astype(np.uint8)


def e2m1_magnitude_code(mag) -> np.ndarray:
    """Index of the nearest E2M1 magnitude; ties go to the even index; beyond 6 saturates."""
    mag = np.asarray(mag, dtype=np.float64)
    d = np.abs(mag[..., None] - E2M1_GRID)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    even = cand & (np.arange(8) % 2 == 0)
    return np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1)).astype(np.uint8)


def mxfp4_quantize_blocks(z) -> tuple[np.ndarray, np.ndarray]:
    """Quantise float32 blocks z[..., 32] -> (4-bit codes[..., 32], E8M0 bytes[...])."""
    z = np.asarray(z, dtype=np.float32)
    amax = np.abs(z).max(axis=-1)
    sbyte = mx_scale_bytes(amax)
    inv_s = np.ldexp(1.0, 127 - sbyte.astype(np.int64))          # 1 / 2^(byte-127), exact
    v = z.astype(np.float64) * inv_s[..., None]                   # exact: power-of-two scaling
    mag = e2m1_magnitude_code(np.abs(v))
    sign = np.signbit(z).astype(np.uint8)
    codes = (sign << 3) | mag
    codes = np.where((amax > 0)[..., None], codes, 0).astype(np.uint8)
    return codes, sbyte


def mxfp4_dequantize_blocks(codes, sbyte) -> np.ndarray:
    """Inverse of the encoding: (-1)^sign * grid[mag] * 2^(byte - 127), in float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = E2M1_GRID[codes & 7]
    sgn = np.where(codes & 8, -1.0, 1.0)
    s = np.ldexp(1.0, np.asarray(sbyte, dtype=np.int64) - 127)
    return sgn * mag * s[..., None]


def pack_nibbles(codes) -> np.ndarray:
    """Two codes per byte along the last axis, the even element in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def quantize_operand(T_bits, hadamard: bool = True, zero_rows=None, zero_cols=None):
    """Residual + (optional) IHT + MXFP4 of an operand laid out lines x J (J = inner dim).

    ``T_bits``: bf16 bit patterns, shape (rows, J).  ``zero_rows`` / ``zero_cols`` are the
    extracted outlier lines, set to +0 before the transform (FOID paragraph: the corresponding
    entries of the residual are zeroed).  Returns (packed codes (rows, J/2) uint8, E8M0 scales
    (rows, J/32) uint8), both J-contiguous.
    """
    x = bf16_to_f32(T_bits).copy()
    rows, J = x.shape
    if J % MX_BLOCK:
        raise ValueError("inner dimension must be a multiple of 32")
    if zero_rows is not None and len(zero_rows):
        x[np.asarray(zero_rows), :] = 0.0
    if zero_cols is not None and len(zero_cols):
        x[:, np.asarray(zero_cols)] = 0.0
    blocks = x.reshape(rows, J // MX_BLOCK, MX_BLOCK)
    if hadamard:
        blocks = fwht32_f32(blocks)
    codes, sbytes = mxfp4_quantize_blocks(blocks)
    return pack_nibbles(codes.reshape(rows, J)), sbytes


def dequantize_operand(packed, sbytes) -> np.ndarray:
    codes = unpack_nibbles(packed)
    rows, J = codes.shape
    return mxfp4_dequantize_blocks(codes.reshape(rows, J // MX_BLOCK, MX_BLOCK),
                                   sbytes).reshape(rows, J)


# --------------------------------------------------------------------------------------------
# FOID (reading R4; Fig. 9 and the appendix FOID paragraph)
# --------------------------------------------------------------------------------------------
def _tree_sum_f32(v: np.ndarray) -> np.ndarray:
    """Sum along the last axis (length 64) by the fixed tree: i + 32, i + 16, ..., i + 1."""
    s = np.asarray(v, dtype=np.float32)
    n = s.shape[-1]
    while n > 1:
        n //= 2
        s = s[..., :n] + s[..., n:2 * n]
    return s[..., 0]


def foid_scores(T_bits, axis: str) -> np.ndarray:
    """float32 population variance of the first 64 elements of every row or column.

    axis="row": line i is row i, probe T[i, 0:64].  axis="col": line j is column j, probe
    T[0:64, j] (the first 64 elements along each column, Fig. 9's red block).
    """
    x = bf16_to_f32(T_bits)
    probe = x[:, :FOID_PROBE] if axis == "row" else x[:FOID_PROBE, :].T
    if probe.shape[1] != FOID_PROBE:
        raise ValueError("lines must hold at least 64 elements")
    sq = (probe * probe).astype(np.float32)     # exact: a bf16 square fits in float32
    s1 = _tree_sum_f32(probe)
    s2 = _tree_sum_f32(sq)
    inv = np.float32(1.0 / FOID_PROBE)
    mean = (s1 * inv).astype(np.float32)
    var = ((s2 * inv).astype(np.float32) - (mean * mean).astype(np.float32)).astype(np.float32)
    return np.where(var > 0, var, np.float32(0.0)).astype(np.float32)


def foid(T_bits, axis: str, r: int) -> np.ndarray:
    """Indices (ascending, int32) of the r lines with the largest probe variance.

    Ranking key: (score bits, then lower index first), so equal scores go to the lower index.
    """
    score = foid_scores(T_bits, axis)
    n = score.shape[0]
    if not 0 <= r <= n:
        raise ValueError("rank out of range")
    key = (score.view(np.uint32).astype(np.uint64) << np.uint64(32)) | \
        (np.uint64(0xFFFFFFFF) - np.arange(n, dtype=np.uint64))
    top = np.sort(key)[::-1][:r]
    lines = (np.uint64(0xFFFFFFFF) - (top & np.uint64(0xFFFFFFFF))).astype(np.int64)
    return np.sort(lines).astype(np.int32)


# --------------------------------------------------------------------------------------------
# Outlier Extraction split (reading R9; appendix FOID paragraph)
# --------------------------------------------------------------------------------------------
def oe_split(T_bits, axis: str, idx):
    """(residual bits with the lines zeroed, outlier lines' original bits).

    axis="row": outlier part is T[idx, :] (r x cols); axis="col": T[:, idx] (rows x r).
    """
    T = np.asarray(T_bits, dtype=np.uint16)
    res = T.copy()
    idx = np.asarray(idx, dtype=np.int64)
    if axis == "row":
        out = T[idx, :].copy()
        res[idx, :] = 0
    else:
        out = T[:, idx].copy()
        res[:, idx] = 0
    return res, out


def oe_merge(res_bits, out_bits, axis: str, idx):
    """Scatter the outlier lines back over the residual (for the exact-reconstruction check)."""
    T = np.asarray(res_bits, dtype=np.uint16).copy()
    idx = np.asarray(idx, dtype=np.int64)
    if axis == "row":
        T[idx, :] = out_bits
    else:
        T[:, idx] = out_bits
    return T


# --------------------------------------------------------------------------------------------
# Calibration and the strategy map (readings R1-R3; abstract, Table 1, Fig. 4, Fig. 5)
# --------------------------------------------------------------------------------------------
def _ratio(s: np.ndarray) -> float:
    med = np.sort(s)[(s.size - 1) // 2]
    top = s.max()
    if med > 0:
        return float(top / med)
    return 1.0 if top == 0 else float("inf")


def calibration_ratios(T_bits) -> tuple[float, float]:
    """(rho_row, rho_col): max / lower-median of the per-row and per-column mean squares."""
    x = bf16_to_f32(T_bits).astype(np.float64)
    sq = x * x
    return _ratio(sq.mean(axis=1)), _ratio(sq.mean(axis=0))


def calibrate_pattern(T_bits, tau: float = DEFAULT_TAU) -> int:
    rho_row, rho_col = calibration_ratios(T_bits)
    if max(rho_row, rho_col) < tau:
        return PAT_NONE
    return PAT_COL if rho_col >= rho_row else PAT_ROW


_PAIR_STRATEGY = {
    (PAT_COL, PAT_NONE): IHT,
    (PAT_NONE, PAT_NONE): IHT,
    (PAT_ROW, PAT_COL): OE_LEFT,
    (PAT_ROW, PAT_NONE): OE_LEFT,
    (PAT_NONE, PAT_COL): OE_RIGHT,
}


def strategy_for_pair(pa: int, pb: int) -> int:
    return _PAIR_STRATEGY.get((pa, pb), BF16)


# GEMM roles.  Fwd: Y = X W^T; dgrad: dX = G_Y W; wgrad: dW = G_Y^T X.  In C = A.B with
# A: P x J and B: J x Q, each source tensor's rows/columns are one of P, Q or J.
SOURCES = {"fwd": ("X", "W"), "dgrad": ("GY", "W"), "wgrad": ("GY", "X")}
AXIS_ROLE = {
    "fwd": {"X": {"row": "P", "col": "J"}, "W": {"row": "Q", "col": "J"}},
    "dgrad": {"GY": {"row": "P", "col": "J"}, "W": {"row": "J", "col": "Q"}},
    "wgrad": {"GY": {"row": "J", "col": "P"}, "X": {"row": "J", "col": "Q"}},
}


def plan_from_patterns(px: int, pw: int, pgy: int, oe_rank: int = DEFAULT_RANK) -> dict:
    pats = {"X": px, "W": pw, "GY": pgy}
    plan = {"patterns": pats, "oe_rank": oe_rank}
    for g in GEMMS:
        a, b = SOURCES[g]
        plan[g] = strategy_for_pair(pats[a], pats[b])
    return plan


def calibrate(X_bits, W_bits, GY_bits, tau: float = DEFAULT_TAU, oe_rank: int = DEFAULT_RANK):
    px = calibrate_pattern(X_bits, tau)
    pw = calibrate_pattern(W_bits, tau)
    pgy = calibrate_pattern(GY_bits, tau) if GY_bits is not None else PAT_NONE
    return plan_from_patterns(px, pw, pgy, oe_rank)


def oe_target(gemm: str, strategy: int, patterns: dict):
    """(source tensor name, line axis) that OE-Left / OE-Right extracts (reading R3)."""
    a, b = SOURCES[gemm]
    if strategy == OE_LEFT:
        rows_wise = [s for s in (a, b) if patterns[s] == PAT_ROW]
        return (rows_wise[0] if len(rows_wise) == 1 else a), "row"
    if strategy == OE_RIGHT:
        cols_wise = [s for s in (a, b) if patterns[s] == PAT_COL]
        return (cols_wise[0] if len(cols_wise) == 1 else b), "col"
    raise ValueError("not an OE strategy")


# --------------------------------------------------------------------------------------------
# The three GEMMs (readings R9-R11; Fig. 5, Fig. 9, appendix GEMM and scatter-add paragraphs)
# --------------------------------------------------------------------------------------------
def gemm_operands(gemm: str, X, W, GY, rows=None, cols=None):
    """bf16 bit views (A: P x J, Bt: Q x J) of one GEMM; Bt is B transposed.  ``rows`` / ``cols``
    (index arrays, or None for all) select lines of A / Bt without forming the others."""
    def take(T, lines, transpose):
        T = np.asarray(T)
        if transpose:
            return np.ascontiguousarray((T if lines is None else T[:, lines]).T)
        return T if lines is None else T[lines]
    if gemm == "fwd":
        return take(X, rows, False), take(W, cols, False)
    if gemm == "dgrad":
        return take(GY, rows, False), take(W, cols, True)
    if gemm == "wgrad":
        return take(GY, rows, True), take(X, cols, True)
    raise ValueError(gemm)


def gemm_plan(gemm: str, strategy: int, patterns: dict, r: int, tensors: dict):
    """Resolve an OE strategy: which operand, which lines, inner or outer.

    Returns None for IHT / MXFP4 / BF16 or r = 0, else a dict with keys
    ``source``, ``axis``, ``idx`` (ascending int32), ``role`` in {"P", "Q", "J"}.
    """
    if strategy not in (OE_LEFT, OE_RIGHT) or r == 0:
        return None
    src, axis = oe_target(gemm, strategy, patterns)
    idx = foid(tensors[src], axis, r)
    return {"source": src, "axis": axis, "idx": idx, "role": AXIS_ROLE[gemm][src][axis]}


def gemm_oracle(gemm: str, strategy: int, X, W, GY, *, patterns=None, r: int = DEFAULT_RANK,
                rows=None, cols=None, oe=None):
    """Everything one AdaHOP GEMM computes, in plain NumPy (float64 for the products).

    ``X`` (M x K), ``W`` (N x K), ``GY`` (M x N) are bf16 bit arrays.  ``rows`` / ``cols``
    restrict the output to a subset of C's rows / columns: every line is quantised on its own
    (its blocks run along J), so only the A lines of the requested rows and the B lines of the
    requested columns are formed and quantised.  ``oe`` may pass a pre-resolved OE plan (as
    returned by ``gemm_plan``; FOID always ranks every line of its source).

    Returns a dict: ``C`` (float64, len(rows) x len(cols)), ``qa``/``qb`` (packed codes, scales)
    of the quantised operand lines, ``oe`` (the resolved OE plan or None), ``a_o``/``b_o`` (inner
    OE slices of those lines, bf16 bits) and ``o`` (outer OE product, float64).
    """
    tensors = {"X": X, "W": W, "GY": GY}
    A, Bt = gemm_operands(gemm, X, W, GY, rows, cols)
    if gemm == "fwd":
        P, Q = np.asarray(X).shape[0], np.asarray(W).shape[0]
    elif gemm == "dgrad":
        P, Q = np.asarray(GY).shape[0], np.asarray(W).shape[1]
    else:
        P, Q = np.asarray(GY).shape[1], np.asarray(X).shape[1]
    rows = np.arange(P) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(Q) if cols is None else np.asarray(cols, dtype=np.int64)
    out = {"oe": None, "qa": None, "qb": None, "a_o": None, "b_o": None, "o": None}

    if strategy == BF16:
        out["C"] = bf16_to_f32(A).astype(np.float64) @ bf16_to_f32(Bt).astype(np.float64).T
        return out

    hadamard = strategy != MXFP4_PLAIN
    if oe is None and strategy in (OE_LEFT, OE_RIGHT):
        oe = gemm_plan(gemm, strategy, patterns, r, tensors)
    out["oe"] = oe

    a_zero_rows = a_zero_cols = b_zero_rows = b_zero_cols = None
    if oe is not None:
        idx = oe["idx"]
        side = "A" if SOURCES[gemm][0] == oe["source"] else "B"
        if oe["role"] == "J":
            if side == "A":
                a_zero_cols = idx
            else:
                b_zero_cols = idx
            out["a_o"] = A[:, idx].copy()           # rows x r, original values
            out["b_o"] = Bt[:, idx].copy()          # cols x r, original values (partner kept)
        elif oe["role"] == "P":
            a_zero_rows = np.nonzero(np.isin(rows, idx))[0]     # positions among the requested rows
        else:  # "Q"
            b_zero_rows = np.nonzero(np.isin(cols, idx))[0]     # positions among the requested columns

    qa = quantize_operand(A, hadamard, zero_rows=a_zero_rows, zero_cols=a_zero_cols)
    qb = quantize_operand(Bt, hadamard, zero_rows=b_zero_rows, zero_cols=b_zero_cols)
    out["qa"], out["qb"] = qa, qb
    C = dequantize_operand(*qa) @ dequantize_operand(*qb).T

    if oe is not None:
        idx = oe["idx"]
        if oe["role"] == "J":
            C = C + bf16_to_f32(out["a_o"]).astype(np.float64) @ bf16_to_f32(out["b_o"]).astype(np.float64).T
        elif oe["role"] == "P":
            A_idx, _ = gemm_operands(gemm, X, W, GY, idx, cols[:0])
            o = bf16_to_f32(A_idx).astype(np.float64) @ bf16_to_f32(Bt).astype(np.float64).T
            out["o"] = o                            # r x len(cols)
            pos = {int(p): i for i, p in enumerate(idx)}
            for k, p in enumerate(rows):
                if int(p) in pos:
                    C[k, :] += o[pos[int(p)]]
        else:
            _, Bt_idx = gemm_operands(gemm, X, W, GY, rows[:0], idx)
            o = bf16_to_f32(A).astype(np.float64) @ bf16_to_f32(Bt_idx).astype(np.float64).T
            out["o"] = o                            # len(rows) x r
            pos = {int(q): i for i, q in enumerate(idx)}
            for k, q in enumerate(cols):
                if int(q) in pos:
                    C[:, k] += o[:, pos[int(q)]]
    out["C"] = C
    return out


def exact_product(gemm: str, X, W, GY, rows=None) -> np.ndarray:
    """A.B over the original bf16 operands in float64 (the quality reference)."""
    A, Bt = gemm_operands(gemm, X, W, GY, None if rows is None else np.asarray(rows))
    return bf16_to_f32(A).astype(np.float64) @ bf16_to_f32(Bt).astype(np.float64).T


def rel_mse(C, C_exact) -> float:
    """||C - C_exact||^2 / ||C_exact||^2 (float64)."""
    C = np.asarray(C, dtype=np.float64)
    E = np.asarray(C_exact, dtype=np.float64)
    return float(((C - E) ** 2).sum() / (E ** 2).sum())


def rel_frobenius(C, C_ref) -> float:
    C = np.asarray(C, dtype=np.float64)
    R = np.asarray(C_ref, dtype=np.float64)
    return float(np.sqrt(((C - R) ** 2).sum() / (R ** 2).sum()))


def iht_improvement(gemm: str, X, W, GY) -> float:
    """Fig. 3's improvement (E_base - E_IHT) / E_base * 100 for one GEMM, where E is the
    relative MSE against the exact product and E_base uses MXFP4 without the Hadamard."""
    exact = exact_product(gemm, X, W, GY)
    e_base = rel_mse(gemm_oracle(gemm, MXFP4_PLAIN, X, W, GY)["C"], exact)
    e_iht = rel_mse(gemm_oracle(gemm, IHT, X, W, GY)["C"], exact)
    return (e_base - e_iht) / e_base * 100.0
