"""Row-band shards of an encoded matrix, for running one product over several
GPUs (one process per GPU).

Tile-row bands are independent in Y = W . X: band b's outputs (rows
b*TM .. b*TM + TM - 1) need only band b's tiles and the whole X.  A shard is a
contiguous range of bands [b0, b1).  Because tile t = tm*nTK + tk numbers the
tiles band-major and the value runs follow the tiles, the shard's bitmap words
and value runs are each ONE contiguous piece of the whole matrix's arrays; only
the offsets need rebasing (the shard's first run starts at element 0).  Every
run is padded to 16 bytes, so a shard's value piece starts on a 16-byte
boundary and can be a view of the original buffer.

X is replicated on every rank; each rank computes its rows of Y (N x M_shard,
token-major), and the rows concatenate along M to the whole result.  Nothing
is exchanged inside a product.  These are host-side steps done once, offline,
like the encoding itself; they work on numpy arrays or torch tensors.
"""
from __future__ import annotations

BITS = {0: 16, 1: 4, 2: 2}            # us_elem -> bits per value


def band_ranges(nTM: int, world: int) -> list[tuple[int, int]]:
    """Contiguous, near-equal ranges of the nTM bands for `world` ranks (a rank
    may get an empty range when world > nTM)."""
    assert nTM >= 0 and world >= 1
    return [(r * nTM // world, (r + 1) * nTM // world) for r in range(world)]


def shard_arrays(bitmap, tile_off, values, M: int, K: int, TM: int, TK: int, elem: int, b0: int, b1: int):
    """Bands [b0, b1) of an encoded matrix.  Returns (bitmap, tile_off, values,
    M_shard): bitmap and values are slices (views) of the inputs, tile_off is a
    new array rebased to start at 0.  tile_off holds uint32 bit patterns (an
    int32 tensor wraps the same way)."""
    nTM, nTK = M // TM, K // TK
    assert 0 <= b0 <= b1 <= nTM
    words = TM * TK // 64
    t0, t1 = b0 * nTK, b1 * nTK
    base = int(tile_off[t0]) & 0xFFFFFFFF
    end = int(tile_off[t1]) & 0xFFFFFFFF
    bits = BITS[elem]
    assert (base * bits) % 128 == 0, "runs are padded to 16 bytes"
    off = tile_off[t0: t1 + 1] - tile_off[t0]
    return bitmap[t0 * words: t1 * words], off, values[base * bits // 8: end * bits // 8], (b1 - b0) * TM


def shard_encoded(E, b0: int, b1: int):
    """An Encoded (device tensors) restricted to bands [b0, b1): bitmap and
    values are views into E's buffers, tile_off a new rebased tensor."""
    from .binding import Encoded
    bm, off, vals, Ms = shard_arrays(E.bitmap, E.tile_off, E.values, E.M, E.K, E.TM, E.TK, E.elem, b0, b1)
    nbytes = vals.numel()
    if nbytes < 16:                     # an empty shard still hands the kernels a valid pointer
        vals = E.values[:16]
    return Encoded(Ms, E.K, E.TM, E.TK, E.elem, E.order, bm, off.contiguous(), vals, nbytes, E.flags)
