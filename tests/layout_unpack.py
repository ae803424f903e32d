"""Host-side reader of the packed cache layout (test utility).

Rebuilds the plain factors of a block, and the window, from the raw bytes of
a cache produced by dkv_compress_layout or dkv_import_factors.  It follows
the layout described in include/dkv.h and csrc/dkv_internal.cuh with its own
index arithmetic (numpy), so a pack -> unpack round trip checks both.
"""
from __future__ import annotations

import numpy as np


def a_layout_index(rows: int, cols: int) -> np.ndarray:
    """Half-element index (in the packed "A layout") of every (row, col): [rows, cols]."""
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    mt, kt = r // 16, c // 16
    rows_in = np.minimum(16, rows - mt * 16)
    cols_in = np.minimum(16, cols - kt * 16)
    nr, nc = rows_in // 8, cols_in // 8
    nsb = nr * nc
    rr, cc = (r % 16) // 8, (c % 16) // 8
    sbi = cc * nr + rr
    lane = (r % 8) * 4 + (c % 8) // 2
    base = mt * 16 * cols * 2 + kt * 16 * rows_in * 2
    byte = base + lane * nsb * 4 + sbi * 4 + (c % 2) * 2
    return byte // 2


def bt_layout_index(rows: int, cols: int) -> np.ndarray:
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    nt, kp = r // 8, c // 32
    lane = (r % 8) * 4 + (c % 8) // 2
    sb = (c % 32) // 8
    byte = nt * 8 * cols * 2 + kp * 512 + lane * 16 + sb * 4 + (c % 2) * 2
    return byte // 2


def exact_index(n_tok: int, d: int) -> tuple[np.ndarray, np.ndarray]:
    """Half-element index of K[t][j] and V[t][j] in a run of 16-token exact groups."""
    K = np.zeros((n_tok, d), np.int64)
    V = np.zeros((n_tok, d), np.int64)
    for g in range(0, n_tok, 16):
        in_g = min(16, n_tok - g)
        gbase = g * 4 * d // 2  # halves: g/16 groups * 64 d bytes
        K[g:g + in_g] = gbase + a_layout_index(in_g, d)
        V[g:g + in_g] = gbase + in_g * d + a_layout_index(d, in_g).T
    return K, V


def is_tc(desc) -> bool:
    """The tensor-core (core-matrix) layout, chosen by the descriptor's `layout` field."""
    return desc.layout == 1


def rd_index(rows: int, d: int) -> np.ndarray:
    """Half-element index of (row, j) of a [rows][d] matrix stored as 8 x 8 core matrices
    (8 rows of 16 bytes each), one plane of d/8 core matrices per 8 rows."""
    r = np.arange(rows)[:, None]
    j = np.arange(d)[None, :]
    byte = (r // 8) * (d // 8) * 128 + (j // 8) * 128 + (r % 8) * 16 + (j % 8) * 2
    return byte // 2


def u_index(r8: int) -> np.ndarray:
    """Half-element index of (token t, r-column k) of U in core matrices: two 128-token
    tiles; inside a tile each 8-token group holds its r8/8 core matrices side by side."""
    t = np.arange(256)[:, None]
    k = np.arange(r8)[None, :]
    byte = (t // 128) * 256 * r8 + ((t % 128) // 8) * 16 * r8 + (k // 8) * 128 + (t % 8) * 16 + (k % 8) * 2
    return byte // 2


def quant_residuals(raw: np.ndarray, n_rows: int, R16: int, d: int, bits: int) -> dict:
    """Codes, fp16 scale and bias of the K and V rows of a block's group-quantised
    residual store (16-token groups: K codes, V^T codes in mma A-fragment order,
    then K scale, K bias, V scale, V bias [d/64][16] fp16), from its raw bytes."""
    G = d // 64
    cb = 16 * d * bits // 8
    gb = 2 * cb + 128 * G
    out = {k: np.zeros((R16, d), np.uint8) for k in ("K_codes", "V_codes")}
    for k in ("K_scale", "K_bias", "V_scale", "V_bias"):
        out[k] = np.zeros((R16, G), np.float16)
    for grp in range(R16 // 16):
        base = grp * gb
        for kv, name in ((0, "K"), (1, "V")):
            words = raw[base + kv * cb: base + (kv + 1) * cb].view(np.uint32)
            for w, word in enumerate(words):
                chunk, lane, wi = w // 128, (w % 128) // 4, w % 4
                gq, t = lane // 4, lane % 4
                for x in range(4 if bits == 8 else 8):
                    if bits == 8:
                        tile, ai, ex, sh, mask = 2 * chunk + wi // 2, 2 * (wi % 2) + x % 2, x // 2, 8 * x, 0xFF
                    else:
                        tile, ai, ex, sh, mask = 4 * chunk + wi, x % 4, x // 4, 4 * x, 0xF
                    r, c = gq + 8 * (ai % 2), 2 * t + ex + 8 * (ai // 2)
                    tok, ch = (16 * grp + r, 16 * tile + c) if kv == 0 else (16 * grp + c, 16 * tile + r)
                    out[name + "_codes"][tok, ch] = (int(word) >> sh) & mask
            sc = raw[base + 2 * cb + kv * 64 * G: base + 2 * cb + (kv + 1) * 64 * G].view(np.float16)
            out[name + "_scale"][16 * grp:16 * grp + 16] = sc[:16 * G].reshape(G, 16).T
            out[name + "_bias"][16 * grp:16 * grp + 16] = sc[16 * G:].reshape(G, 16).T
    for k in list(out):
        out[k] = out[k][:n_rows] if k.endswith(("codes", "scale", "bias")) else out[k]
    return out


def unpack_block(cache: np.ndarray, desc, u: int, b: int) -> dict:
    d, r, r8, R, R8 = desc.head_dim, desc.rank, desc.rank_pad, desc.n_residual, desc.res_pad
    unit = u * desc.unit_stride
    blk = unit + desc.off_blocks + b * desc.block_stride
    h = lambda off, n: cache[off:off + 2 * n].view(np.float16)
    tc = is_tc(desc)
    out = {}
    out["a_k"] = h(blk, d).copy()
    out["a_v"] = h(blk + 2 * d, d).copy()
    words = cache[blk + desc.blk_off_mask: blk + desc.blk_off_mask + 32].view(np.uint32)
    out["mask"] = np.array([(words[i >> 5] >> (i & 31)) & 1 for i in range(256)], dtype=bool)
    vk = h(blk + desc.blk_off_vk, r8 * d)
    out["V_K"] = vk[bt_layout_index(r8, d)][:r].copy()
    uu = h(blk + desc.blk_off_u, 256 * r8)
    Ufull = uu[u_index(r8)]  # both layouts store U as 8 x 8 core matrices
    out["U_row0"] = Ufull[0].copy()
    out["U"] = Ufull[1:, :r].copy()
    if desc.residual_bits:
        q = quant_residuals(cache[blk + desc.blk_off_res: blk + desc.blk_off_vv], R, R8, d, desc.residual_bits)
        out.update(q)
        deq = lambda c, s, bb: (c.astype(np.float64).reshape(R, d // 64, 64) * s.astype(np.float64)[:, :, None]
                                + bb.astype(np.float64)[:, :, None]).reshape(R, d)
        out["K_res"] = deq(q["K_codes"], q["K_scale"], q["K_bias"])
        out["V_res"] = deq(q["V_codes"], q["V_scale"], q["V_bias"])
        res = None
    else:
        res = h(blk + desc.blk_off_res, 2 * R8 * d)
    if res is None:
        pass
    elif tc:
        ki = rd_index(R8, d)
        vi = R8 * d + ki
    else:
        ki, vi = exact_index(R8, d)
    if res is not None:
        out["K_res"] = res[ki][:R].copy()
        out["V_res"] = res[vi][:R].copy()
        out["res_pad_zero"] = bool((res[ki][R:] == 0).all() and (res[vi][R:] == 0).all())
    vv = h(blk + desc.blk_off_vv, r8 * d)
    out["V_V"] = (vv[rd_index(r8, d)] if tc else vv[a_layout_index(d, r8)].T)[:r].copy()
    if desc.rope_dims:  # un-rotated pool: fp32 boxes of the rotated keys, 8d bytes a block
        off = unit + desc.off_router + b * 8 * d
        router = cache[off:off + 8 * d].view(np.float32)
    else:
        router = h(unit + desc.off_router + b * 4 * d, 2 * d)
    out["kmin"], out["kmax"] = router[:d].copy(), router[d:].copy()
    cold = cache[unit + desc.off_cold + b * R8 * 2: unit + desc.off_cold + (b + 1) * R8 * 2].view(np.uint16)
    out["S"] = cold[:R].astype(np.int64)
    return out


def unpack_window(cache: np.ndarray, desc, u: int) -> tuple[np.ndarray, np.ndarray]:
    d, W, W16 = desc.head_dim, desc.window, desc.window_pad
    off = u * desc.unit_stride + desc.off_window
    win = cache[off: off + W16 * 4 * d].view(np.float16)
    if is_tc(desc):
        ki = np.zeros((W16, d), np.int64)
        vi = np.zeros((W16, d), np.int64)
        for g in range(0, W16, 128):
            n = min(128, W16 - g)
            base = g * 4 * d // 2          # halves: 128-token groups of K then V
            ki[g:g + n] = base + rd_index(n, d)
            vi[g:g + n] = base + n * d + rd_index(n, d)
    else:
        ki, vi = exact_index(W16, d)
    return win[ki][:W].copy(), win[vi][:W].copy()


def unpack_rope_tables(cache: np.ndarray, desc) -> tuple[np.ndarray, np.ndarray]:
    """The un-rotated pool's RoPE tables: page entries [pages][h] and in-page entries
    [256][h], each (cos, sin) as fp32."""
    h = desc.rope_dims // 2
    n = (desc.total_bytes - desc.off_rope) // (8 * h)
    tab = cache[desc.off_rope:desc.off_rope + n * h * 8].view(np.float32).reshape(n, h, 2)
    return tab[:n - 256], tab[n - 256:]
