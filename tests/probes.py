"""Inputs placed at and next to the rounding midpoints of the quantiser's
decisions, for a tensor scale g (shared by the oracle pins and the GPU tests).

Every builder returns BF16 bit patterns or raw pool bytes; expected values are
left to the caller (exact rational rounding on the CPU, the oracle on the GPU).
"""

from fractions import Fraction as Fr

import numpy as np

import oracle
from exact_rounding import E2M1, E4M3, bf16_neighbours, bf16_rne_bits, bf16_value, rne_code

E4M3_MIDS = [(E4M3[c] + E4M3[c + 1]) / 2 for c in range(126)]
E2M1_MIDS = [(E2M1[c] + E2M1[c + 1]) / 2 for c in range(7)]


def f32(x) -> float:
    return float(np.float32(x))


def fp32_scale_code(amax_bits, g):
    """The FP32 shortcut the exact rule replaces: E4M3(fl32(amax / fl32(6 g)))."""
    q = np.float32(bf16_value(amax_bits)) / (np.float32(6.0) * np.float32(g))
    return rne_code(Fr(float(q)), E4M3)


def scale_traps(n_wanted=4):
    """(g, amax bits, exact scale code) next to amax / (6 mid) for BF16 amax and
    E4M3 midpoints, where the FP32 quotient decides another code than exact rounding."""
    found = []
    for ci in range(40, 126, 3):
        mid = E4M3_MIDS[ci]
        for a_bits in bf16_neighbours(6 * mid * Fr(3, 7), 2):
            a = bf16_value(a_bits)
            g = np.float32(float(a / (6 * mid)))
            cands = [g]
            for direction in (np.float32(np.inf), np.float32(-np.inf)):
                h = g
                for _ in range(3):
                    h = np.nextafter(h, direction)
                    cands.append(h)
            for gc in cands:
                gc = float(gc)
                exact = rne_code(a / (6 * Fr(gc)), E4M3)
                if exact != fp32_scale_code(a_bits, gc):
                    found.append((gc, a_bits, exact))
                    if len(found) >= n_wanted:
                        return found
    return found


def product_traps(n_wanted=3):
    """Tensor scales g for which some e2m1 * e4m3 * g, rounded to FP32 first, lands
    on a BF16 midpoint that the exact product is not on, on the side that makes
    BF16(FP32(.)) differ from BF16 of the exact product."""
    mags = sorted({E2M1[c] * E4M3[s] for c in range(1, 8) for s in range(1, 127)})
    found = []
    rng = np.random.default_rng(5)
    for _ in range(4000):
        p = mags[int(rng.integers(len(mags)))]
        g0 = Fr(float(np.float32(2.0 ** rng.uniform(-3, 3))))
        m_bits = bf16_rne_bits(p * g0) & 0x7FFF
        mid = (bf16_value(m_bits) + bf16_value(m_bits + 1)) / 2
        g = f32(float(mid / p))
        fp32 = Fr(float(np.float32(float(p)) * np.float32(g)))
        if fp32 == mid and bf16_rne_bits(fp32) != bf16_rne_bits(p * Fr(g)):
            found.append(g)
            if len(found) >= n_wanted:
                break
    return found


G_SET = [f32(0.3), f32(3.7), 1.5, 0.75, f32(1.0 / 2688), f32(2.0**-110 * 1.37), f32(2.0**90 * 1.9),
         f32(2.0**-126), f32(3.0e38)]


def block(first_bits, rest_bits=()):
    x = np.zeros(16, dtype=np.uint16)
    x[0] = first_bits
    for i, b in enumerate(rest_bits):
        x[1 + i] = b
    return x


def scale_probe_blocks(g):
    """Blocks whose amax (element 0, either sign) lies at and next to 6 g mid for
    every E4M3 midpoint mid, and past saturation."""
    G = Fr(g)
    out = []
    for mid in E4M3_MIDS + [E4M3[126] * Fr(33, 32)]:
        for a_bits in bf16_neighbours(6 * G * mid, 2):
            for neg in (0, 0x8000):
                out.append(block(a_bits | neg))
    return np.array(out)


def amax_for_scale(sc, G):
    """A BF16 amax whose exact scale decision at G is code sc, or None."""
    for a_bits in bf16_neighbours(6 * G * E4M3[sc], 1):
        if rne_code(bf16_value(a_bits) / (6 * G), E4M3) == sc:
            return a_bits
    return None


def code_probe_blocks(g, scales=None):
    """Blocks with a known scale s (element 0 the amax that yields it) whose 15
    other elements, alternating in sign, lie at and next to mid * s * g for every
    E2M1 midpoint mid and past saturation.  Returns (blocks, their scale codes)."""
    G = Fr(g)
    blocks, codes = [], []
    for sc in (scales if scales is not None else list(range(1, 127, 5)) + [8, 56, 125, 126]):
        a_bits = amax_for_scale(sc, G)
        if a_bits is None:
            continue
        amax = bf16_value(a_bits)
        den = E4M3[sc] * G
        cands = []
        for mid in E2M1_MIDS + [E2M1[7] * Fr(17, 16)]:
            cands += [b for b in bf16_neighbours(mid * den, 1) if bf16_value(b) <= amax]
        for i in range(0, len(cands), 15):
            chunk = cands[i:i + 15]
            blocks.append(block(a_bits, [c | ((j % 2) << 15) for j, c in enumerate(chunk)]))
            codes.append(sc)
    return np.array(blocks), codes


def fp8_probe_values(g):
    """BF16 values (alternating in sign) at and next to mid * g for every E4M3
    midpoint mid and past saturation."""
    G = Fr(g)
    xs = []
    for mid in E4M3_MIDS + [E4M3[126] * Fr(33, 32)]:
        xs += bf16_neighbours(mid * G, 1)
    xs = np.array(sorted(set(xs)), dtype=np.uint16)
    xs[1::2] |= 0x8000
    return xs


def rows_of(values, width=128):
    """Pad a flat uint16 array with zeros to whole rows [n][1][width]."""
    v = np.asarray(values, dtype=np.uint16).reshape(-1)
    n = -(-len(v) // width)
    out = np.zeros(n * width, dtype=np.uint16)
    out[:len(v)] = v
    return out.reshape(n, 1, width)


def all_products():
    """(e2m1 code, e4m3 code) pairs over every E2M1 code and every finite E4M3 scale."""
    return [(c, s) for s in list(range(0, 127)) + list(range(128, 255)) for c in range(16)]


def crafted_pool(dtype, g, P=16):
    """An oracle pool (one kv head) whose K and V rows hold every (E2M1 code,
    E4M3 scale) pair (NVFP4: block b of row r holds 16 codes sharing one scale)
    or every finite E4M3 code (FP8), written at the documented offsets.
    Returns (pool, rows used)."""
    assert P == 16
    if dtype == oracle.DTYPE_NVFP4:
        pairs = all_products()
        blocks = -(-len(pairs) // 16)
        rows = -(-blocks // 8)
        pool = oracle.OraclePool(-(-rows // P), P, 1, gk=g, gv=g)
        for blk in range(blocks):
            r, b = divmod(blk, 8)
            page, rr = divmod(r, P)          # P = 16: one 16-row group per page
            chunk = pairs[blk * 16:(blk + 1) * 16]
            codes = [c for c, _ in chunk]
            packed = [codes[2 * i] | (codes[2 * i + 1] << 4) for i in range(8)]
            # K codes [16][64] | K scales [16][8] | V codes [16][64] | V scales [8][16]
            for code_off, scale_off in ((rr * 64 + b * 8, 1024 + rr * 8 + b),
                                        (1152 + rr * 64 + b * 8, 2176 + b * 16 + rr)):
                pool.data[page, 0, code_off:code_off + 8] = packed
                pool.data[page, 0, scale_off] = chunk[0][1]
        return pool, rows
    codes = list(range(0, 127)) + list(range(128, 255))
    rows = -(-len(codes) // 128)
    pool = oracle.OraclePool(-(-rows // P), P, 1, dtype=oracle.DTYPE_FP8, gk=g, gv=g)
    for i, c in enumerate(codes):
        r, d = divmod(i, 128)
        page, rr = divmod(r, P)
        for which in (0, 1):                 # K codes [16][128] | V codes [16][128]
            pool.data[page, 0, which * 2048 + rr * 128 + d] = c
    return pool, rows
