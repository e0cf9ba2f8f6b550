"""IO-complexity model of the pages, pinned by their worked numbers.
Test infrastructure only (see the package docstring).

[FA-notes] §3.5 Theorem 2: standard attention needs Theta(N d + N^2) HBM
accesses, the tiled algorithm Theta(N^2 d^2 / M) for SRAM size M (in
elements); the notes evaluate both at N = 1024, d = 64, M = 25,600 fp32.
[FA-notes] §2.1 / §3.3 and [S12] "问题" give the size of a materialised
N x N score/probability matrix.
"""
from __future__ import annotations


def standard_hbm_accesses(N: int, d: int) -> int:
    """Theta(N d + N^2) with unit constant ([FA-notes] §3.5)."""
    return N * d + N * N


def flash_hbm_accesses(N: int, d: int, M: int) -> float:
    """Theta(N^2 d^2 / M) with unit constant ([FA-notes] §3.5)."""
    return N * N * d * d / M


def materialized_matrix_bytes(N: int, bytes_per_elem: int, n_matrices: int = 1,
                              heads: int = 1) -> int:
    """Bytes of ``n_matrices`` materialised N x N matrices over ``heads`` heads."""
    return n_matrices * heads * N * N * bytes_per_elem

