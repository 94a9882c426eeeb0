"""Oracle for the FP8 linear-layer hot path: plain, slow, obviously correct, CPU only.

TEST INFRASTRUCTURE. Only the tests, the package smoke check and the benchmark's CPU-baseline
leg may import this module. It shares no code with the CUDA path and imports nothing from it.

Sources. The recipes are those of the Megatron Core developer guide page "Low-Precision
Training Guide" (sections "Hardware and Recipe Compatibility", "Recipe Reference" with its
delayed / tensorwise / mxfp8 / blockwise entries, and "Numerical Stability Knobs"), the
TransformerEngine issue "How to reduce cuda memory usage of fp8?" (which FP8 copies the
backward pass caches), and the MegaDLMs summary "Benefits of Using FP8 Precision with
MegaDLMs and Required Hardware" (activation_func_fp8_input_store, --no-fp8-wgrad).
The pages name the recipes, block shapes, history knobs and margin but print no formulas;
where they are silent the readings below are the plainest ones the rest supports:

  * E4M3 is the OCP 8-bit "E4M3FN" format: bias 7, no infinities, 0x7F/0xFF NaN,
    max 448 (0x7E), min subnormal 2^-9 (0x01). Encoding rounds to nearest, ties to even,
    and saturates finite overflow and +-inf to +-448; -0 keeps its sign.
  * The "hybrid" format (--fp8-format hybrid, delayed / tensorwise / blockwise only) keeps
    activations and weights in E4M3 and stores gradients in E5M2, the OCP 8-bit format with
    bias 15, two mantissa bits, +-inf at 0x7C/0xFC, NaN 0x7D-0x7F, max 57344 (0x7B), min
    subnormal 2^-16 (0x01). It is encoded like E4M3 (round to nearest even, finite overflow
    and +-inf saturate to +-57344, NaN -> 0x7F with the input's sign) and its scales use
    57344 in place of 448.
  * Per-tensor scale (tensorwise, delayed, and per block for blockwise):
    s = fp32(448 / amax) * 2^-margin, one IEEE fp32 division; s = 1 when amax is 0 or not
    finite; an infinite s is clamped to FLT_MAX; the stored dequantisation factor is
    s_inv = fp32(1 / s). The margin is M bits of extra headroom (Numerical Stability Knobs).
  * A code is encode(fp32(x * s)): the product is rounded to fp32 first, then to E4M3.
  * MXFP8: per 1x32 block the E8M0 exponent is the smallest e with amax <= 448 * 2^e,
    clamped to [-127, 127]; blocks with amax below 2^-126 (zero, or subnormal) get -127.
    The stored byte is e + 127. Codes are encode(x * 2^-e), an exact product. A block
    holding an Inf or a NaN gets the E8M0 NaN byte 0xFF and codes encode(x) (e = 0).
  * Delayed: the history starts as L zeros and s = 1; a step quantises with the scale from
    the history of the previous steps only, then pushes its own amax (evicting the oldest
    entry once L are held) and derives the next scale from max(history).
  * Power-of-two block scales (the blockwise recipe's option that maps onto power-of-two
    hardware scaling): the block scale above is rounded down to a power of two.
  * Blockwise: 1x128 blocks for activations and gradients, whose column-wise copy is
    re-quantised from bf16 with 1x128 blocks along the other dimension; 128x128 blocks for
    weights, whose column-wise copy is the byte transpose with the scale grid transposed.
  * GEMMs: every code is decoded and multiplied by its dequantisation factor in float64, the
    product is summed in float64 (numpy matmul), and the result is rounded once to bf16.
  * GeLU is the exact form h * Phi(h) (Phi evaluated through erfc so the negative tail keeps
    full relative precision); its derivative is Phi(h) + h * phi(h).

Conventions: X[M,K] activations, W[N,K] weights, Y = X W^T, dY[M,N]. The row-wise copy
has the source's shape with blocks along its last dimension; the column-wise copy is the
transposed tensor with blocks along its own last dimension. bf16 tensors are numpy uint16
bit patterns; codes are uint8; scales are float32 (per-tensor, 1x128, 128x128) or uint8
E8M0 bytes (MXFP8).

Parity pins: every function here is pinned by a test in tests/test_oracle_*.py against an
independent fact (torch's own float8 conversion, brute force over the 254 finite codes,
exact rational matmuls on small inputs, hand-computed scale sequences, closed forms).
"""
import math

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6      # smallest normal binade: [2^-6, 2^-5)
E4M3_MANTISSA_BITS = 3
E5M2_MAX = 57344.0
E5M2_MIN_NORMAL_EXP = -14
E5M2_MANTISSA_BITS = 2
FP8_MAX = {"e4m3": E4M3_MAX, "e5m2": E5M2_MAX}
FLT_MAX = np.float32(np.finfo(np.float32).max)
MX_BLOCK = 32
BW_BLOCK = 128


# --------------------------------------------------------------------------------------
# bf16 storage
# --------------------------------------------------------------------------------------

def bf16_to_f32(bits):
    """bf16 bit patterns -> float32 (exact widening: bf16 is the upper half of float32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def as_f32(x):
    """A quantiser's input as float32 values: bf16 bit patterns (uint16) are widened exactly;
    float32 arrays (fp32 master weights, cast without a bf16 rounding) pass through."""
    x = np.asarray(x)
    if x.dtype == np.float32:
        return x
    if x.dtype == np.uint16:
        return bf16_to_f32(x)
    raise TypeError("quantiser input: bf16 bit patterns (uint16) or float32")


def f64_to_bf16(v):
    """float64 -> bf16 bit pattern, one rounding to nearest, ties to even, on the bf16 grid.

    Written from the definition: bf16 has 8 significant bits and the float32 exponent
    range, so the quantum of a value in binade [2^E, 2^(E+1)) is 2^(E-7) (2^-133 below the
    smallest normal). Values beyond the largest bf16 round to +-inf; NaN stays NaN.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    a = np.abs(v)
    sign = np.signbit(v)
    _, ex = np.frexp(a)
    E = np.maximum(ex - 1, -126)
    quantum = np.ldexp(1.0, E - 7)
    r = np.rint(a / quantum) * quantum          # exact: power-of-two quantum
    max_bf16 = float(np.ldexp(255.0, 120))      # (2 - 2^-7) * 2^127
    r = np.where(r > max_bf16, np.inf, r)
    f = r.astype(np.float32)                    # exact: r is on the bf16 grid (or inf)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(sign, bits | np.uint16(0x8000), bits)
    out[...] = np.where(np.isnan(v), np.uint16(0x7FC0), bits)
    return out


# --------------------------------------------------------------------------------------
# E4M3 (OCP E4M3FN)
# --------------------------------------------------------------------------------------

def e4m3_decode(codes):
    """E4M3 codes -> float64 values: e == 0 gives m * 2^-9, else (1 + m/8) * 2^(e-7)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = s * mag
    return np.where((e == 15) & (m == 7), np.nan, val)


def e4m3_encode(v):
    """float32 values -> E4M3 codes, round to nearest with ties to even, saturating.

    The value's binade [2^E, 2^(E+1)) (E never below -6, the subnormal range) fixes the
    quantum 2^(E-3); the magnitude is divided by it and rounded half-to-even to an integer
    count n. n * quantum is then an E4M3 value (a count of 16 is the carry into the next
    binade). Magnitudes >= 448, including infinity, give 448; NaN gives the NaN code.
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    sign = np.where(np.signbit(v), 0x80, 0x00).astype(np.int64)
    nan = np.isnan(v)
    sat = (a >= E4M3_MAX) & ~nan
    a_ok = np.where(sat | nan, 0.0, a)

    _, ex = np.frexp(a_ok)                       # a = f * 2^ex, f in [0.5, 1)
    E = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, E - E4M3_MANTISSA_BITS)
    n = np.rint(a_ok / quantum)                  # numpy rint: round half to even
    val = n * quantum                            # the chosen E4M3 magnitude, <= 448

    # fields of val
    _, vex = np.frexp(val)
    vE = vex - 1
    normal = val >= 2.0 ** E4M3_MIN_NORMAL_EXP
    e_field = np.where(normal, vE + 7, 0)
    m_field = np.where(normal,
                       np.rint((val / np.ldexp(1.0, np.where(normal, vE, 0)) - 1.0) * 8.0),
                       np.rint(val / 2.0 ** -9))
    code = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    code = np.where(sat, 0x7E, code)
    code = np.where(nan, 0x7F, code)
    return (code | sign).astype(np.uint8)


# --------------------------------------------------------------------------------------
# E5M2 (OCP E5M2), the gradient format of the hybrid recipe
# --------------------------------------------------------------------------------------

def e5m2_decode(codes):
    """E5M2 codes -> float64: e == 0 gives m * 2^-16, e == 31 gives +-inf (m = 0) or NaN,
    else (1 + m/4) * 2^(e-15)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 2) & 0x1F
    m = c & 0x3
    mag = np.where(e == 0, m * 2.0 ** -16, (1.0 + m / 4.0) * np.ldexp(1.0, e - 15))
    mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    return s * mag


def e5m2_encode(v):
    """float32 values -> E5M2 codes, round to nearest with ties to even, saturating.

    As for E4M3: the binade [2^E, 2^(E+1)) (E never below -14) has the quantum 2^(E-2); the
    magnitude is rounded half-to-even to a count of quanta (a count of 8 carries into the next
    binade). Magnitudes >= 57344, infinity included, give 57344; NaN gives 0x7F (with sign).
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    sign = np.where(np.signbit(v), 0x80, 0x00).astype(np.int64)
    nan = np.isnan(v)
    sat = (a >= E5M2_MAX) & ~nan
    a_ok = np.where(sat | nan, 0.0, a)
    _, ex = np.frexp(a_ok)
    E = np.maximum(ex - 1, E5M2_MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, E - E5M2_MANTISSA_BITS)
    val = np.rint(a_ok / quantum) * quantum      # an E5M2 magnitude, <= 57344
    _, vex = np.frexp(val)
    vE = vex - 1
    normal = val >= 2.0 ** E5M2_MIN_NORMAL_EXP
    e_field = np.where(normal, vE + 15, 0)
    m_field = np.where(normal,
                       np.rint((val / np.ldexp(1.0, np.where(normal, vE, 0)) - 1.0) * 4.0),
                       np.rint(val / 2.0 ** -16))
    code = (e_field.astype(np.int64) << 2) | m_field.astype(np.int64)
    code = np.where(sat, 0x7B, code)
    code = np.where(nan, 0x7F, code)
    return (code | sign).astype(np.uint8)


def fp8_encode(v, fmt="e4m3"):
    return e5m2_encode(v) if fmt == "e5m2" else e4m3_encode(v)


def fp8_decode(codes, fmt="e4m3"):
    return e5m2_decode(codes) if fmt == "e5m2" else e4m3_decode(codes)


def hybrid_format(role):
    """Format of a tensor under --fp8-format hybrid: gradients E5M2, the rest E4M3."""
    return "e5m2" if role == "grad" else "e4m3"


# --------------------------------------------------------------------------------------
# Per-tensor scale (tensorwise, delayed; per block for blockwise)
# --------------------------------------------------------------------------------------

def pow2_floor(s):
    """Largest power of two <= s for positive finite float32 s (exact, through the exponent);
    0 stays 0."""
    s = np.asarray(s, dtype=np.float32).astype(np.float64)
    _, ex = np.frexp(s)                           # s = f * 2^ex, f in [0.5, 1)
    return np.where(s > 0, np.ldexp(1.0, ex - 1), 0.0).astype(np.float32)


def scales_from_amax(amax, margin=0, fmt="e4m3", pow2=False):
    """(s, s_inv) as float32 arrays from amax values: s = fp32(448/amax) * 2^-margin, s_inv = 1/s
    (57344 in place of 448 for E5M2). With pow2 (power-of-two block scales), s is then rounded
    down to a power of two, so s_inv is exact and no element can exceed the format's maximum.

    The tensorwise entry derives the scale from the tensor being cast; --fp8-margin
    (Numerical Stability Knobs) gives the scale M extra bits of headroom. The division
    is one IEEE fp32 division; the 2^-margin factor is applied exactly in float64 and the
    result narrowed once to fp32; amax 0 or non-finite gives s = 1; infinite s -> FLT_MAX.
    """
    a = np.asarray(amax, dtype=np.float32)
    ok = np.isfinite(a) & (a != 0)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        s = np.where(ok, np.float32(FP8_MAX[fmt]) / np.where(ok, a, np.float32(1.0)),
                     np.float32(1.0)).astype(np.float32)
        s = np.ldexp(s.astype(np.float64), -int(margin)).astype(np.float32)
    s = np.where(np.isinf(s), FLT_MAX, s).astype(np.float32)
    if pow2:
        s = pow2_floor(s)
    s_inv = (np.float32(1.0) / s).astype(np.float32)
    return s, s_inv


def scale_from_amax(amax, margin=0, fmt="e4m3"):
    """Scalar form of scales_from_amax: returns (s, s_inv) as numpy float32 scalars."""
    s, s_inv = scales_from_amax(np.float32(amax), margin, fmt)
    return np.float32(s), np.float32(s_inv)


def amax_of(x_bf16):
    """max |x| over a bf16 (or float32) tensor, as float32 (exact). NaN if any element is NaN."""
    x = as_f32(x_bf16)
    if x.size == 0:
        return np.float32(0.0)
    return np.float32(np.max(np.abs(x)))


def cast_with_scale(x_bf16, s, fmt="e4m3"):
    """codes = encode(fp32(x * s)): one fp32 product, then the FP8 rounding."""
    x = as_f32(x_bf16)
    return fp8_encode((x * np.float32(s)).astype(np.float32), fmt)


def quantize_tensorwise(x_bf16, margin=0, fmt="e4m3"):
    """Tensorwise current scaling (recipe entry "tensorwise").

    Returns dict(amax, scale, scale_inv, row=[R,C] codes, col=[C,R] codes); the column-wise
    copy is the byte transpose of the row-wise copy (one scale for the whole tensor).
    """
    amax = amax_of(x_bf16)
    s, s_inv = scale_from_amax(amax, margin, fmt)
    row = cast_with_scale(x_bf16, s, fmt)
    return dict(amax=amax, scale=s, scale_inv=s_inv, row=row, col=np.ascontiguousarray(row.T))


# --------------------------------------------------------------------------------------
# Delayed scaling (recipe entry "delayed")
# --------------------------------------------------------------------------------------

class DelayedScaling:
    """Rolling amax history of length L with the `max` (or `most_recent`) compute algorithm.

    --fp8-amax-history-len L, --fp8-amax-compute-algo {max, most_recent}, --fp8-margin M.
    The page's minimum config names `max`; `most_recent` is the knob's other setting (the
    newest amax alone decides the next scale).
    """

    def __init__(self, history_len, margin=0, fmt="e4m3", algo="max"):
        if history_len < 1:
            raise ValueError("amax history length must be >= 1")
        if algo not in ("max", "most_recent"):
            raise ValueError("amax compute algo is max or most_recent")
        self.L = int(history_len)
        self.margin = int(margin)
        self.fmt = fmt
        self.algo = algo
        self.history = np.zeros(self.L, dtype=np.float32)
        self.head = 0
        self.scale = np.float32(1.0)
        self.scale_inv = np.float32(1.0)

    def quantize(self, x_bf16):
        """Quantise with the current scale; return codes and this tensor's amax."""
        amax = amax_of(x_bf16)
        row = cast_with_scale(x_bf16, self.scale, self.fmt)
        return dict(amax=amax, scale=self.scale, scale_inv=self.scale_inv, row=row,
                    col=np.ascontiguousarray(row.T))

    def update(self, amax_new):
        """Push amax_new (oldest entry evicted) and derive the next scale from the window's max
        (`max`) or from amax_new alone (`most_recent`, the history is still recorded)."""
        self.history[self.head] = np.float32(amax_new)
        self.head = (self.head + 1) % self.L
        a = np.max(self.history) if self.algo == "max" else np.float32(amax_new)
        self.scale, self.scale_inv = scale_from_amax(a, self.margin, self.fmt)
        return self.scale, self.scale_inv


# --------------------------------------------------------------------------------------
# MXFP8 (recipe entry "mxfp8": one power-of-two scale for each 1x32 block of E4M3 data)
# --------------------------------------------------------------------------------------

def mx_exponent(amax_block):
    """Smallest integer e with amax <= 448 * 2^e (clamped to [-127, 127]); -127 below 2^-126.

    With amax = m * 2^E, m in [1, 2): 448 = 1.75 * 2^8, so e = E - 8 when m <= 1.75 and
    E - 7 when m > 1.75. Works element-wise on float32 arrays, in exact integer steps.
    """
    a = np.asarray(amax_block, dtype=np.float32).astype(np.float64)
    tiny = ~(a >= 2.0 ** -126)                    # zero, subnormal (and NaN: treated as tiny)
    f, ex = np.frexp(np.where(tiny, 1.0, a))      # a = f * 2^ex, f in [0.5, 1)
    m = 2.0 * f
    E = ex - 1
    e = E - 8 + (m > 1.75).astype(np.int64)
    e = np.clip(e, -127, 127)
    return np.where(tiny, -127, e).astype(np.int64)


def _mx_quantize_lastdim(x_f32):
    """MX-quantise along the last dim of a float32 [R, C]: codes [R,C], E8M0 bytes [R,C/32]."""
    R, C = x_f32.shape
    blocks = x_f32.reshape(R, C // MX_BLOCK, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    bad = ~np.isfinite(amax)                      # the block holds an Inf or a NaN
    e = np.where(bad, 0, mx_exponent(np.where(bad, 0.0, amax)))
    scaled = blocks.astype(np.float64) * np.ldexp(1.0, -e)[:, :, None]   # exact
    codes = e4m3_encode(scaled.astype(np.float32)).reshape(R, C)
    return codes, np.where(bad, 255, e + 127).astype(np.uint8)


def quantize_mxfp8(x_bf16, want_col=True):
    """Row-wise copy with 1x32 blocks along C, column-wise copy of X^T with blocks along R.

    Returns dict(row=[R,C], row_scale=[R,C/32], col=[C,R], col_scale=[C,R/32]); the column
    entries are omitted when want_col is False (the row copy of any subset of rows is then
    the same as that subset of the full tensor's row copy).
    """
    x = as_f32(x_bf16)
    row, row_scale = _mx_quantize_lastdim(x)
    out = dict(row=row, row_scale=row_scale)
    if want_col:
        out["col"], out["col_scale"] = _mx_quantize_lastdim(np.ascontiguousarray(x.T))
    return out


def e8m0_decode(bytes_):
    """E8M0 byte b -> 2^(b-127) as float64 (0xFF would be NaN; the quantiser never emits it)."""
    b = np.asarray(bytes_, dtype=np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


# --------------------------------------------------------------------------------------
# Blockwise (recipe entry "blockwise": 1x128 activation blocks, 128x128 weight blocks)
# --------------------------------------------------------------------------------------

def _bw_quantize_1x128_lastdim(x_bf16, margin, fmt="e4m3", pow2=False):
    """Per 1x128 block along the last dim: codes [R,C], s_inv [R, C/128] (float32)."""
    x = as_f32(x_bf16)
    R, C = x.shape
    blocks = x.reshape(R, C // BW_BLOCK, BW_BLOCK)
    s, s_inv = scales_from_amax(np.max(np.abs(blocks), axis=2), margin, fmt, pow2)
    codes = fp8_encode((blocks * s[:, :, None]).astype(np.float32), fmt).reshape(R, C)
    return codes, s_inv


def quantize_blockwise_1x128(x_bf16, margin=0, fmt="e4m3", pow2=False):
    """Activations / gradients: row copy with 1x128 blocks along C, column copy of X^T
    re-quantised from bf16 with 1x128 blocks along R.

    Returns dict(row=[R,C], row_scale_inv=[R,C/128], col=[C,R], col_scale_inv=[C,R/128]).
    """
    x = as_f32(x_bf16)
    row, row_si = _bw_quantize_1x128_lastdim(x, margin, fmt, pow2)
    col, col_si = _bw_quantize_1x128_lastdim(np.ascontiguousarray(x.T), margin, fmt, pow2)
    return dict(row=row, row_scale_inv=row_si, col=col, col_scale_inv=col_si)


def quantize_blockwise_128x128(x_bf16, margin=0, fmt="e4m3", pow2=False):
    """Weights: one scale per 128x128 tile; column copy = byte transpose, grid transposed.

    Returns dict(row=[R,C], row_scale_inv=[R/128, C/128], col=[C,R], col_scale_inv=[C/128,R/128]).
    """
    x = as_f32(x_bf16)
    R, C = x.shape
    gr, gc = R // BW_BLOCK, C // BW_BLOCK
    tiles = x.reshape(gr, BW_BLOCK, gc, BW_BLOCK)            # [i, r, j, c]
    s, s_inv = scales_from_amax(np.max(np.abs(tiles), axis=(1, 3)), margin, fmt, pow2)
    codes = fp8_encode((tiles * s[:, None, :, None]).astype(np.float32), fmt).reshape(R, C)
    return dict(row=codes, row_scale_inv=s_inv, col=np.ascontiguousarray(codes.T),
                col_scale_inv=np.ascontiguousarray(s_inv.T))


def pow2_scales_as_e8m0(s_inv, block_rows, rows, cols):
    """Power-of-two block scales written as MXFP8 E8M0 bytes [rows][cols/32]: a power-of-two
    s_inv = 2^k is exactly the E8M0 byte k + 127, repeated for the four 1x32 blocks of each
    128-wide block (and, for 128x128 tiles, for the tile's 128 rows). s_inv is [rows][cols/128]
    for 1x128 blocks (block_rows 1) or [rows/128][cols/128] for 128x128 tiles."""
    s = np.asarray(s_inv, dtype=np.float32).astype(np.float64)
    f, ex = np.frexp(s)
    if not np.all(f == 0.5):
        raise ValueError("not a power-of-two scale")
    b = (ex - 1 + 127).astype(np.int64)
    b = np.repeat(b, 4, axis=1)
    if block_rows == 128:
        b = np.repeat(b, 128, axis=0)
    assert b.shape == (rows, cols // 32)
    return b.astype(np.uint8)


# --------------------------------------------------------------------------------------
# Dequantisation and the fp64 GEMM reference
# --------------------------------------------------------------------------------------

def dequant_tensor(codes, scale_inv, fmt="e4m3"):
    """Per-tensor: decode(code) * s_inv, in float64."""
    return fp8_decode(codes, fmt) * np.float64(np.float32(scale_inv))


def dequant_mx(codes, e8m0):
    """MXFP8 along the last dim: decode(code) * 2^(b-127) for the element's 1x32 block."""
    f = np.repeat(e8m0_decode(e8m0), MX_BLOCK, axis=1)
    return e4m3_decode(codes) * f


def dequant_1x128(codes, s_inv, fmt="e4m3"):
    """1x128 blocks along the last dim: decode(code) * s_inv of the element's block."""
    f = np.repeat(np.asarray(s_inv, dtype=np.float32).astype(np.float64), BW_BLOCK, axis=1)
    return fp8_decode(codes, fmt) * f


def dequant_128x128(codes, s_inv, fmt="e4m3"):
    """128x128 tiles: decode(code) * s_inv of the element's tile."""
    f = np.asarray(s_inv, dtype=np.float32).astype(np.float64)
    f = np.repeat(np.repeat(f, BW_BLOCK, axis=0), BW_BLOCK, axis=1)
    return fp8_decode(codes, fmt) * f


def gemm_tn_f64(a_deq, b_deq):
    """C[m,n] = sum_k A[m,k] * B[n,k] in float64 (both operands K-major, as every GEMM of
    the layer is: fprop X.W^T, dgrad dY.(W^T)^T, wgrad (dY^T).(X^T)^T)."""
    return np.asarray(a_deq, dtype=np.float64) @ np.asarray(b_deq, dtype=np.float64).T


def gemm_tn_f64_rows(a_deq, b_deq, rows):
    """The same sum for a subset of output rows (sampled parity at full size)."""
    return gemm_tn_f64(np.asarray(a_deq)[rows], b_deq)


def bf16_gemm_tn_f64(a_bf16, b_bf16):
    """The bf16 wgrad path (--fp8-wgrad False): the same fp64 sum over bf16 operands."""
    return gemm_tn_f64(bf16_to_f32(a_bf16).astype(np.float64),
                       bf16_to_f32(b_bf16).astype(np.float64))


# --------------------------------------------------------------------------------------
# GeLU with its input stored in FP8 (activation_func_fp8_input_store)
# --------------------------------------------------------------------------------------

_erfc = np.vectorize(math.erfc, otypes=[np.float64])


def normal_cdf(h):
    """Phi(h) = 0.5 erfc(-h / sqrt 2): the same function as 0.5 (1 + erf(h / sqrt 2)), but
    without the cancellation that formula suffers when erf is close to -1 (h below about -5)."""
    return 0.5 * _erfc(-np.asarray(h, dtype=np.float64) / math.sqrt(2.0))


def gelu_f64(h):
    """gelu(h) = h Phi(h) = 0.5 h (1 + erf(h / sqrt 2)), float64."""
    h = np.asarray(h, dtype=np.float64)
    return h * normal_cdf(h)


def gelu_grad_f64(h):
    """gelu'(h) = Phi(h) + h phi(h), float64."""
    h = np.asarray(h, dtype=np.float64)
    phi = np.exp(-0.5 * h * h) / math.sqrt(2.0 * math.pi)
    return normal_cdf(h) + h * phi


def gelu_bf16(h_bf16):
    """a = bf16(gelu(h)) from a bf16 h."""
    return f64_to_bf16(gelu_f64(bf16_to_f32(h_bf16)))


def dgelu_bf16(da_bf16, h_codes, h_e8m0):
    """dh = bf16(da * gelu'(deq(h_fp8))): the backward reads h back from its FP8 copy."""
    h = dequant_mx(h_codes, h_e8m0)
    return f64_to_bf16(bf16_to_f32(da_bf16).astype(np.float64) * gelu_grad_f64(h))
