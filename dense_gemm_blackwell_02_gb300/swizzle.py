"""Model of the 128-byte shared-memory swizzle used by the operand ring and
the epilogue staging tile.

"A Blackwell GEMM by Hand in CuTe DSL", section 6: with 128-byte rows, the
16-byte chunk index (address bits 4..6) is XORed with the row index modulo 8
(address bits 7..9).  A row keeps its bytes; only the order of its eight
chunks changes.  The CUDA epilogue writes its staging tile in this layout so
that a TMA store with CU_TENSOR_MAP_SWIZZLE_128B reads it back in row order.

Shared memory has 32 banks of 4 bytes; a 16-byte access covers 4 banks.
`bank_passes` counts the serialised wavefronts a set of 16-byte accesses
needs: the largest number of distinct 4-byte words that land in one bank.
"""
from __future__ import annotations

CHUNK = 16
ROW = 128
BANKS = 32


def sw128(byte_addr: int) -> int:
    """Physical byte address of logical `byte_addr` under the 128B swizzle."""
    row = (byte_addr // ROW) % 8
    chunk = (byte_addr // CHUNK) % 8
    return byte_addr - chunk * CHUNK + ((chunk ^ row) * CHUNK)


def bank_passes(chunk_addrs) -> int:
    words_in_bank = [set() for _ in range(BANKS)]
    for a in chunk_addrs:
        first = a // 4
        for w in range(first, first + CHUNK // 4):
            words_in_bank[w % BANKS].add(w)
    return max(len(s) for s in words_in_bank)


def column_passes(tile_k: int, elem_bytes: int = 2, swizzled: bool = False):
    """Passes for reading one 16-byte column chunk from 8 consecutive rows of
    a tile whose rows are tile_k elements long, for every chunk of the row.
    Returns None when the 128B swizzle does not apply (rows shorter than 128 B)."""
    pitch = tile_k * elem_bytes
    if swizzled and pitch < ROW:
        return None
    f = sw128 if swizzled else (lambda a: a)
    return [bank_passes([f(r * pitch + c * CHUNK) for r in range(8)])
            for c in range(pitch // CHUNK)]


def sw128_chunk_permutation(row: int):
    """Physical chunk positions of logical chunks 0..7 in the given row."""
    return [(sw128(row * ROW + c * CHUNK) - row * ROW) // CHUNK for c in range(8)]
