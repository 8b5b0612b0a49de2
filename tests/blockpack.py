"""Test-side packer for hand-built expert blobs in the canonical block layout.

Writes integer codes into bytes following the pages' bit order (code n of a Q2_0
block in bits 2(n%4).. of byte n/4; Q4 nibble n in bits 4(n%2).. of byte n/2),
each block prefixed by its fp16 scale. Used only to build inputs whose layer
output has a closed form; the decoding side is pinned by the golden fixtures.
"""
import numpy as np

Q4, Q2 = 0, 1


def block_weights(kind):
    return 64 if kind == Q2 else 32


def pack_matrix(kind, codes, scales):
    """codes: int [rows][cols] (0..3 or 0..15); scales: float [rows][cols/bw] -> bytes."""
    codes = np.asarray(codes, dtype=np.int64)
    rows, cols = codes.shape
    bw = block_weights(kind)
    nb = cols // bw
    scales = np.broadcast_to(np.asarray(scales, dtype=np.float64), (rows, nb))
    out = np.zeros((rows, nb, 18), dtype=np.uint8)
    sb = scales.astype(np.float16).view(np.uint16)
    out[:, :, 0] = sb & 0xFF
    out[:, :, 1] = sb >> 8
    for r in range(rows):
        for b in range(nb):
            blk = codes[r, b * bw:(b + 1) * bw]
            cb = np.zeros(16, dtype=np.int64)
            for n, q in enumerate(blk):
                if kind == Q2:
                    cb[n // 4] |= int(q) << (2 * (n % 4))
                else:
                    cb[n // 2] |= int(q) << (4 * (n % 2))
            out[r, b, 2:] = cb.astype(np.uint8)
    return out.reshape(-1)


def pack_expert(kind, gate_codes, up_codes, down_codes, gate_scale, up_scale, down_scale):
    return np.concatenate([pack_matrix(kind, gate_codes, gate_scale),
                           pack_matrix(kind, up_codes, up_scale),
                           pack_matrix(kind, down_codes, down_scale)])


def selector_expert(kind, zp, H, F, pi, sigma, rho, a_code, b_code, c_code, dg=1.0, du=1.0, dd=1.0):
    """Expert whose gate row f picks x[pi[f]] (weight dg*(a_code-zp)), up row f picks
    x[sigma[f]] (du*(b_code-zp)), down column f writes h[f] to output rho[f]
    (dd*(c_code-zp)); every other weight is 0 (code zp)."""
    g = np.full((F, H), zp)
    u = np.full((F, H), zp)
    d = np.full((H, F), zp)
    for f in range(F):
        g[f, pi[f]] = a_code
        u[f, sigma[f]] = b_code
        d[rho[f], f] = c_code
    return pack_expert(kind, g, u, d, dg, du, dd)
