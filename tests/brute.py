"""Pure-Python brute force used to pin the C oracle on tiny inputs.

Written independently of oracle/us_oracle.c: bit strings instead of shifts,
Python integers instead of fixed-width arithmetic, ``fractions`` for exact sums.
Format rules restated (UnionSparse section V-A with one area; SPDP section 4.1
column tiles and the 16-byte padding of its section 4.2.3):
tile t = tm*nTK + tk; scan row-major (ROW) or column-major (COL) inside the tile;
bit for scan position p is bit p%64 of word p//64, earlier positions in lower
bits; nonzeros appended in scan order; each tile's run padded with zeros to a
multiple of 8 fp16, 32 int4 or 64 int2 elements (int2: four per byte, the
earlier element in the lower bits, two's complement); offsets count elements.
"""
from fractions import Fraction

import numpy as np


def scan_positions(TM, TK, order):
    if order == 0:
        return [(i, j) for i in range(TM) for j in range(TK)]
    return [(i, j) for j in range(TK) for i in range(TM)]


def encode(W, TM, TK, elem, order):
    """W: list of lists of ints (int4 codes) or of uint16 fp16 bit patterns."""
    M, K = len(W), len(W[0])
    quantum = {0: 8, 1: 32, 2: 64}[elem]
    words, offsets, stream = [], [0], []
    for tm in range(M // TM):
        for tk in range(K // TK):
            bits = ""
            for (i, j) in scan_positions(TM, TK, order):
                v = W[tm * TM + i][tk * TK + j]
                nz = (v & 0x7FFF) != 0 if elem == 0 else v != 0
                bits += "1" if nz else "0"
                if nz:
                    stream.append(v)
            for q in range(0, len(bits), 64):
                chunk = bits[q:q + 64]
                words.append(int(chunk[::-1], 2))    # position 0 -> least significant bit
            run = len(stream) - offsets[-1]
            while run % quantum:
                stream.append(0)
                run += 1
            offsets.append(len(stream))
    if elem == 0:
        data = b"".join(int(v).to_bytes(2, "little") for v in stream)
    elif elem == 1:
        nib = [(v + 16) % 16 for v in stream]
        data = bytes(nib[k] + 16 * nib[k + 1] for k in range(0, len(nib), 2))
    else:
        cr = [(v + 4) % 4 for v in stream]
        data = bytes(cr[k] + 4 * cr[k + 1] + 16 * cr[k + 2] + 64 * cr[k + 3] for k in range(0, len(cr), 4))
    return words, offsets, data


def dot_w4a4(wrow, xrow):
    return sum(int(a) * int(b) for a, b in zip(wrow, xrow))


def dot_f16_exact(wrow, xrow):
    """Exact rational sum of fp16 products."""
    return sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(wrow, xrow))


def to_lists(a: np.ndarray):
    return [[int(v) for v in row] for row in a]
