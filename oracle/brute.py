"""fp64 brute force: dequantise every block to real values, then plain matmuls.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is a second,
independent restatement of the block formats (vectorised numpy, numpy's own
binary16 conversion, the E2M1 magnitudes as real numbers rather than the
doubled integer lattice) used to pin the integer-dot oracle in ``oracle.c``:
the integer/scale factoring there must reproduce these dense fp64 products
to within fp64 rounding.

Formats (GGUF-style blocks; element value in terms of the stored fields):
  Q8_0 : {f16 d; i8 q[32]}                 w = d q
  Q4_K : {f16 d; f16 dmin; u8 s[12]; u8 qs[128]}
         w = d sc_j q - dmin m_j over 8 sub-blocks of 32; 6-bit (sc, m) packed
         in s (j<4: low 6 bits of s[j], s[j+4]; j>=4: nibbles of s[j+4] plus
         the top 2 bits of s[j-4], s[j]); qs byte 32g+l holds element 64g+l in
         its low nibble and 64g+32+l in its high nibble.
  Q2_K : {u8 s[16]; u8 qs[64]; f16 d; f16 dmin}
         w = d sc_j q - dmin m_j over 16 sub-blocks of 16, sc = s[j] & 15,
         m = s[j] >> 4; bits 2s..2s+1 of qs[32n+l] give element 128n+32s+l.
  MXFP4: {u8 e; u8 qs[16]}                 w = 2^(e-127) * E2M1(code)
         code of element j < 16 is the low nibble of qs[j], of j+16 the high
         nibble; bit 3 is the sign.
  Q6_K : {u8 ql[128]; u8 qh[64]; i8 sc[16]; f16 d}
         w = d sc_j (c - 32) over 16 sub-blocks of 16, c a 6-bit code: for
         element 128n+32s+l its low nibble is nibble s//2 of ql[64n+32(s%2)+l]
         and its top 2 bits are bits 2s..2s+1 of qh[32n+l].
  Q3_K : {u8 hmask[32]; u8 qs[64]; u8 sc[12]; f16 d}
         w = d (s_j - 32) c over 16 sub-blocks of 16, c = (2 bits at 2s of
         qs[32n+l]) - 4 * (1 - bit 4n+s of hmask[l]); 6-bit s_j: nibble j//8
         of byte j%8 plus 2 high bits at 2(j//4) of byte 8 + j%4.
"""
from __future__ import annotations

import numpy as np

F32, Q8_0, Q4_K, Q2_K, MXFP4, Q6_K, Q3_K = 0, 1, 2, 3, 4, 5, 6
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)


def _f16(b: np.ndarray) -> np.ndarray:
    """little-endian byte pairs [..., 2] -> float64 via numpy's binary16."""
    return np.ascontiguousarray(b).view(np.float16)[..., 0].astype(np.float64)


def dequant(qtype: int, blocks: np.ndarray, cols: int) -> np.ndarray:
    """uint8 [rows, row_bytes] -> float64 [rows, cols]."""
    if qtype == F32:
        return np.ascontiguousarray(blocks).view(np.float32).astype(np.float64).reshape(-1, cols)
    rows = blocks.shape[0]
    if qtype == Q8_0:
        b = blocks.reshape(rows, cols // 32, 34)
        d = _f16(b[..., 0:2])
        q = b[..., 2:].view(np.int8).astype(np.float64)
        return (d[..., None] * q).reshape(rows, cols)
    if qtype == Q4_K:
        b = blocks.reshape(rows, cols // 256, 144)
        d, dm = _f16(b[..., 0:2]), _f16(b[..., 2:4])
        s = b[..., 4:16].astype(np.int64)
        sc = np.empty(b.shape[:2] + (8,), np.int64)
        mn = np.empty_like(sc)
        sc[..., :4] = s[..., 0:4] & 63
        mn[..., :4] = s[..., 4:8] & 63
        sc[..., 4:] = (s[..., 8:12] & 15) | ((s[..., 0:4] >> 6) << 4)
        mn[..., 4:] = (s[..., 8:12] >> 4) | ((s[..., 4:8] >> 6) << 4)
        qs = b[..., 16:].astype(np.int64).reshape(rows, -1, 4, 32)      # [.., g, l]
        q = np.concatenate([qs & 15, qs >> 4], axis=-1)                 # [.., g, 64]
        q = q.reshape(rows, -1, 8, 32).astype(np.float64)               # sub-block j = 2g + (hi)
        w = d[..., None, None] * sc[..., None] * q - dm[..., None, None] * mn[..., None]
        return w.reshape(rows, cols)
    if qtype == Q2_K:
        b = blocks.reshape(rows, cols // 256, 84)
        s = b[..., 0:16].astype(np.int64)
        sc, mn = s & 15, s >> 4
        qs = b[..., 16:80].astype(np.int64).reshape(rows, -1, 2, 1, 32)  # [.., n, 1, l]
        sh = np.arange(4).reshape(1, 1, 1, 4, 1) * 2
        q = ((qs >> sh) & 3).reshape(rows, -1, 16, 16).astype(np.float64)  # element 128n+32s+l
        d, dm = _f16(b[..., 80:82]), _f16(b[..., 82:84])
        w = d[..., None, None] * sc[..., None] * q - dm[..., None, None] * mn[..., None]
        return w.reshape(rows, cols)
    if qtype == MXFP4:
        b = blocks.reshape(rows, cols // 32, 17)
        scale = np.ldexp(1.0, b[..., 0].astype(np.int64) - 127)
        qs = b[..., 1:].astype(np.int64)
        code = np.concatenate([qs & 15, qs >> 4], axis=-1)
        mag = _E2M1[code & 7]
        val = np.where(code & 8, -mag, mag)
        return (scale[..., None] * val).reshape(rows, cols)
    if qtype == Q6_K:
        b = blocks.reshape(rows, cols // 256, 210).astype(np.int64)
        ql = b[..., 0:128].reshape(rows, -1, 2, 2, 32)                  # [.., n, s%2, l]
        qh = b[..., 128:192].reshape(rows, -1, 2, 1, 32)                # [.., n, 1, l]
        lo = np.concatenate([ql & 15, ql >> 4], axis=-2)                # [.., n, s, l], s = 2*(nibble) + s%2
        hi = (qh >> (2 * np.arange(4).reshape(4, 1))) & 3
        code = (lo | (hi << 4)) - 32
        sc = blocks.reshape(rows, cols // 256, 210)[..., 192:208].view(np.int8).astype(np.float64)
        d = _f16(blocks.reshape(rows, cols // 256, 210)[..., 208:210])
        w = d[..., None, None] * sc[..., None] * code.reshape(rows, -1, 16, 16).astype(np.float64)
        return w.reshape(rows, cols)
    if qtype == Q3_K:
        raw = blocks.reshape(rows, cols // 256, 110)
        b = raw.astype(np.int64)
        hm = b[..., 0:32].reshape(rows, -1, 1, 1, 32)
        qs = b[..., 32:96].reshape(rows, -1, 2, 1, 32)
        s = np.arange(4).reshape(1, 4, 1)
        n = np.arange(2).reshape(2, 1, 1)
        code = ((qs >> (2 * s)) & 3) - 4 * (1 - ((hm >> (4 * n + s)) & 1))   # [.., n, s, l]
        s12 = b[..., 96:108]
        low = np.concatenate([s12[..., 0:8] & 15, s12[..., 0:8] >> 4], axis=-1)
        high = np.stack([(s12[..., 8:12] >> (2 * g)) & 3 for g in range(4)], axis=-2).reshape(rows, -1, 16)
        scale = ((low | (high << 4)) - 32).astype(np.float64)
        d = _f16(raw[..., 108:110])
        w = d[..., None, None] * scale[..., None] * code.reshape(rows, -1, 16, 16).astype(np.float64)
        return w.reshape(rows, cols)
    raise ValueError(qtype)


def act_values(d: np.ndarray, q: np.ndarray) -> np.ndarray:
    """q8 activations -> float64 values: d broadcast over its block of codes."""
    T, n = q.shape
    B = n // d.shape[1]
    return (np.repeat(d.astype(np.float64), B, axis=1) * q.astype(np.float64))


def silu(g):
    return g / (1.0 + np.exp(-g))


def expert_gu(layer, e: int, xv: np.ndarray, shared: bool = False):
    """g, u [T, I] for expert e (or the shared expert) on activation values xv [T, H]."""
    cfg = layer.cfg
    if shared:
        qt, gate, up, bg, bu = cfg.shared_qtype, layer.sgate[0], layer.sup[0], None, None
    else:
        qt, gate, up = cfg.qtype, layer.gate[e], layer.up[e]
        bg = None if layer.bg is None else layer.bg[e].astype(np.float64)
        bu = None if layer.bu is None else layer.bu[e].astype(np.float64)
    Wg, Wu = dequant(qt, gate, cfg.H), dequant(qt, up, cfg.H)
    g, u = xv @ Wg.T, xv @ Wu.T
    if bg is not None:
        g = g + bg
    if bu is not None:
        u = u + bu
    return g, u


def expert_o(layer, e: int, hv: np.ndarray, shared: bool = False):
    """o [T, H] for expert e on requantised-h values hv [T, I]."""
    cfg = layer.cfg
    if shared:
        Wd = dequant(cfg.shared_qtype, layer.sdown[0], cfg.shared_I)
        return hv @ Wd.T
    Wd = dequant(cfg.qtype, layer.down[e], cfg.I)
    o = hv @ Wd.T
    if layer.bd is not None:
        o = o + layer.bd[e].astype(np.float64)
    return o


def ffn_given_hq(layer, xq, ids, w, hq_slots, hq_shared=None):
    """y [T, H] in fp64 using the requantised h supplied per (token, slot).

    hq_slots: (hd [T, k, I/B], hq [T, k, I]) ; hq_shared: (hd [T, Is/B], hq [T, Is])."""
    cfg = layer.cfg
    T, k = ids.shape
    xv = act_values(xq[0], xq[1])
    y = np.zeros((T, cfg.H), np.float64)
    for t in range(T):
        for s in range(k):
            e = int(ids[t, s])
            hv = act_values(hq_slots[0][t, s][None], hq_slots[1][t, s][None])
            y[t] += w[t, s] * expert_o(layer, e, hv)[0]
        if hq_shared is not None:
            hv = act_values(hq_shared[0][t][None], hq_shared[1][t][None])
            y[t] += expert_o(layer, 0, hv, shared=True)[0]
    return y
