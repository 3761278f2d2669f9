"""Counter-based generator of bf16 ~N(0,1) values.

Every value is a pure function of a 64-bit key that packs
(seed, workload, stream, layer, frame, tensor, token, head, d):

    bits  0..5   d        (head_dim <= 64)
    bits  6..10  head     (heads <= 32)
    bits 11..24  token    (token index inside its frame, < 16384)
    bits 25..26  tensor   (0 = q, 1 = k, 2 = v, 3 = schedule draws)
    bits 27..42  frame    (< 65536)
    bits 43..47  layer    (< 32)
    bits 48..53  stream   (< 64)
    bits 54..56  workload (< 8)
    bits 57..63  seed     (< 128)

The key is hashed with splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are
Vigna's published 64-bit variant): z = key + 0x9E3779B97F4A7C15, then two
xor-shift-multiply rounds and a final xor-shift.

The 64-bit hash is cut into four 16-bit uniforms u1..u4 (low half first).
Their Irwin-Hall sum has mean 131070 and variance 2^32/3, so

    x = fl32( fl32(u1+u2+u3+u4 - 131070) * 2^-16 ) * fl32(1.7320508)

has unit variance. The first product is exact (an integer below 2^18 scaled
by a power of two), the second is one IEEE fp32 round-to-nearest-even
multiply. An optional power-of-two scale (queries use 2^-3) is exact too.
The result is rounded to bf16 with round-to-nearest-even. Each step is exact
or a single correctly-rounded operation, so any faithful IEEE implementation
(numpy here, the CUDA generator kernel on the device) gives the same bits.
"""

import numpy as np

TENSOR_Q = 0
TENSOR_K = 1
TENSOR_V = 2
TENSOR_DRAW = 3

_M64 = (1 << 64) - 1
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MUL1 = np.uint64(0xBF58476D1CE4E5B9)
_MUL2 = np.uint64(0x94D049BB133111EB)


def pack_key(seed, workload, stream, layer, frame, tensor, token, head, d):
    """Pack the generator's coordinates into one 64-bit key (numpy uint64,
    broadcasting over array arguments). Raises if a field is out of range."""
    fields = ((seed, 7, 57), (workload, 3, 54), (stream, 6, 48), (layer, 5, 43),
              (frame, 16, 27), (tensor, 2, 25), (token, 14, 11), (head, 5, 6),
              (d, 6, 0))
    key = np.uint64(0)
    for value, width, shift in fields:
        arr = np.asarray(value, dtype=np.int64)
        if arr.size and (arr.min() < 0 or arr.max() >= (1 << width)):
            raise ValueError(f"generator key field out of range: width {width}, shift {shift}")
        key = key | (arr.astype(np.uint64) << np.uint64(shift))
    return key


def splitmix64(key):
    """splitmix64 output for state `key` (uint64 arrays wrap modulo 2^64)."""
    with np.errstate(over="ignore"):
        z = np.asarray(key, dtype=np.uint64) + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MUL1
        z = (z ^ (z >> np.uint64(27))) * _MUL2
        return z ^ (z >> np.uint64(31))


def _f32_to_bf16_bits(x):
    """Round fp32 to bf16 (round-to-nearest-even) and return the 16-bit patterns.
    The generator never produces NaN or inf."""
    bits = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def gaussian_bf16(keys, scale=1.0):
    """bf16 bit patterns (uint16) of the ~N(0,1) value for each key, times `scale`
    (must be a power of two so that the scaling is exact)."""
    h = splitmix64(keys)
    s = np.zeros(h.shape, dtype=np.int64)
    for i in range(4):
        s += ((h >> np.uint64(16 * i)) & np.uint64(0xFFFF)).astype(np.int64)
    x = (s - 131070).astype(np.float32) * np.float32(2.0 ** -16)
    x = x * np.float32(1.7320508)
    if scale != 1.0:
        m, _ = np.frexp(scale)
        if m != 0.5:
            raise ValueError("scale must be a power of two")
        x = x * np.float32(scale)
    return _f32_to_bf16_bits(x)


def frame_tensor(seed, workload, stream, layer, frame, tensor, n_tokens, heads, head_dim,
                 scale=1.0, token0=0):
    """One frame's q, k or v as bf16 bits, layout [n_tokens][heads][head_dim]."""
    tok = np.arange(token0, token0 + n_tokens, dtype=np.int64)[:, None, None]
    hh = np.arange(heads, dtype=np.int64)[None, :, None]
    dd = np.arange(head_dim, dtype=np.int64)[None, None, :]
    keys = pack_key(seed, workload, stream, layer, frame, tensor, tok, hh, dd)
    return gaussian_bf16(keys, scale)


def uniform_draw(seed, workload, stream, index):
    """A raw 64-bit draw for workload schedules (stream lengths, intervals)."""
    return int(splitmix64(pack_key(seed, workload, stream, 0, 0, TENSOR_DRAW, index, 0, 0)))


def bf16_bits_to_f32(bits):
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits):
    """Exact widening of bf16 bit patterns to fp64."""
    return bf16_bits_to_f32(bits).astype(np.float64)
