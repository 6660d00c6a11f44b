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
    out = []
    for r in range(rows_pad):
        for b in range(na * 4):
            if r < rows and b < nb:
                continue
            atom = (r // 128) * na + b // 4
            out.append(buf[off + atom * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)])
    return np.array(out, np.uint8)
