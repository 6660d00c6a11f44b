"""Test-side reading of the rs operand device layout documented in
include/rs.h, written independently of librs: maps the device buffer back to
the oracle's logical arrays (codes [rows][K/2], scales [rows][K/bs])."""
import numpy as np


def block_size(fmt):
    return 16 if fmt == 0 else 32


def sf_offset(rows, K):
    return (rows * (K // 2) + 1023) // 1024 * 1024


def n_atoms_k(fmt, K):
    ak = 4 * block_size(fmt)
    return (K + ak - 1) // ak


def operand_bytes(fmt, rows, K):
    return sf_offset(rows, K) + (rows + 127) // 128 * n_atoms_k(fmt, K) * 512


def unpack_operand(buf, fmt, rows, K):
    """buf: uint8 numpy array of the whole operand."""
    buf = np.asarray(buf, np.uint8)
    codes = buf[: rows * (K // 2)].reshape(rows, K // 2)
    off = sf_offset(rows, K)
    nb = K // block_size(fmt)
    na = n_atoms_k(fmt, K)
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    atom = (r // 128) * na + b // 4
    idx = off + atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return codes.copy(), buf[idx]


def padding_sf_bytes(buf, fmt, rows, K):
    """Scale bytes of the padding rows / padding blocks (must be zero)."""
    buf = np.asarray(buf, np.uint8)
    off = sf_offset(rows, K)
    na = n_atoms_k(fmt, K)
    rows_pad = (rows + 127) // 128 * 128
    nb = K // block_size(fmt)
    r = np.arange(rows_pad)[:, None]
    b = np.arange(na * 4)[None, :]
    pad = (r >= rows) | (b >= nb)
    atom = (r // 128) * na + b // 4
    idx = off + atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return buf[idx[pad]]


def weight_block_bytes(fmt):
    return 16384 + (4 if fmt == 0 else 2) * 512


def weight_bytes(fmt, N, K):
    return (N + 127) // 128 * ((K + 255) // 256) * weight_block_bytes(fmt)


def unpack_weight(buf, fmt, N, K):
    """rs weight (tiled, swizzled) -> logical codes [N][K/2], scales [N][K/bs];
    also returns whether every padding byte is zero."""
    buf = np.asarray(buf, np.uint8)
    wb = weight_block_bytes(fmt)
    nt, nc = (N + 127) // 128, (K + 255) // 256
    blocks = buf[: nt * nc * wb].reshape(nt, nc, wb)
    codes_img = blocks[:, :, :16384].reshape(nt, nc, 128, 128)
    r = np.arange(128)[:, None]
    j = np.arange(128)[None, :]
    src = ((j // 16) ^ (r % 8)) * 16 + j % 16           # position of byte j of row r
    codes_full = np.take_along_axis(codes_img, np.broadcast_to(src, codes_img.shape), axis=3)
    codes_full = codes_full.transpose(0, 2, 1, 3).reshape(nt * 128, nc * 128)
    bs = block_size(fmt)
    apb = 256 // (4 * bs)                                  # atoms per block
    atoms = blocks[:, :, 16384:].reshape(nt, nc, apb, 512)
    nb_full = nc * 256 // bs
    rr = np.arange(nt * 128)[:, None]
    bb = np.arange(nb_full)[None, :]
    t = rr // 128
    c = bb // (256 // bs)
    a = (bb % (256 // bs)) // 4
    off = (rr % 32) * 16 + ((rr % 128) // 32) * 4 + bb % 4
    sf_full = atoms[t, c, a, off]
    codes = codes_full[:N, : K // 2].copy()
    sf = sf_full[:N, : K // bs].copy()
    pad_ok = (not codes_full[N:].any() and not codes_full[:, K // 2:].any()
              and not sf_full[N:].any() and not sf_full[:, K // bs:].any())
    return codes, sf, pad_ok


# ---- paged NVFP4 KV cache (decode attention) ----
# Page p of KV head h: codes [32 tokens][D/2] then E4M3 scales [32][D/16];
# pages stored [page][Hkv]; a block table [B][max_pages] maps each sequence's
# logical pages (token t -> page block_table[b][t // 32], row t % 32).

PAGE = 32


def page_bytes(D):
    return PAGE * (D // 2 + D // 16)


def pack_paged_cache(codes, sf, seq_lens, rng=None):
    """Logical codes [B][L][Hkv][D/2] and scales [B][L][Hkv][D/16] -> (cache
    bytes [n_pages][Hkv][page_bytes], block table int32 [B][max_pages]).
    Pages are handed out in a shuffled order so the table is not trivial;
    rows past a sequence's length stay zero."""
    codes = np.asarray(codes, np.uint8)
    sf = np.asarray(sf, np.uint8)
    B, L, H, CB = codes.shape
    SB = sf.shape[3]
    D = 2 * CB
    max_pages = (L + PAGE - 1) // PAGE
    need = [(int(n) + PAGE - 1) // PAGE for n in seq_lens]
    order = np.arange(sum(need))
    if rng is not None:
        rng.shuffle(order)
    cache = np.zeros((max(len(order), 1), H, page_bytes(D)), np.uint8)
    table = np.zeros((B, max_pages), np.int32)
    k = 0
    for b in range(B):
        for lp in range(need[b]):
            page = int(order[k])
            k += 1
            table[b, lp] = page
            t0, t1 = lp * PAGE, min(int(seq_lens[b]), (lp + 1) * PAGE)
            for h in range(H):
                blk = cache[page, h]
                rows = t1 - t0
                blk[:rows * CB] = codes[b, t0:t1, h].reshape(-1)
                blk[PAGE * CB:PAGE * CB + rows * SB] = sf[b, t0:t1, h].reshape(-1)
    return cache, table


def unpack_paged_cache(cache, table, seq_lens, D):
    """Inverse of pack_paged_cache on the first seq_lens[b] tokens."""
    cache = np.asarray(cache, np.uint8)
    B = table.shape[0]
    H = cache.shape[1]
    CB, SB = D // 2, D // 16
    L = table.shape[1] * PAGE
    codes = np.zeros((B, L, H, CB), np.uint8)
    sf = np.zeros((B, L, H, SB), np.uint8)
    for b in range(B):
        for t in range(int(seq_lens[b])):
            blk = cache[table[b, t // PAGE]]
            r = t % PAGE
            codes[b, t] = blk[:, r * CB:(r + 1) * CB]
            sf[b, t] = blk[:, PAGE * CB + r * SB:PAGE * CB + (r + 1) * SB]
    return codes, sf
