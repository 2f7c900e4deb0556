"""One emulated DGEMM split into output blocks over the ranks of a process group.

[Q] "誤差のないINT8行列積(手順3)": the N residue products are independent, the
residues and the reconstruction are per entry, and the scaling is per row of A
and per column of B.  So the ranks form a pr x pc grid; rank (a, b) owns the
row block a of A (and of C) and the column block b of B (and of C) and
computes C[rows_a, cols_b] with the library's kernels on its own GPU.

- Fast mode: the exponent of row i depends on row i alone (and that of column
  j on column j alone), so every rank runs os2_gemm on its block: no
  collective, and C is identical, entry for entry, to the unsplit product's.
- Accurate mode: the bound R_i is the maximum of row i of the bound product
  over all columns, and K_j of column j over all rows.  Each rank computes its
  block's maxima (os2_scale_bounds); a MAX-allreduce over the ranks of the same
  row block gives R, one over the ranks of the same column block gives K
  (m + n int32 per rank in all); then the exponents (os2_exponents_from_bounds)
  and steps 2-5 (os2_gemm_exponents) run locally.  C is again identical to the
  unsplit product's.

The collective is torch.distributed (NCCL between GPUs; gloo for the CPU
tests of the same grid and reduction code).  Argument marshalling and the
split only: every step of the method runs in the library's kernels.
"""
from __future__ import annotations

import math

import torch
import torch.distributed as dist


def grid_shape(world: int) -> tuple[int, int]:
    """The most nearly square pr x pc = world grid (pr <= pc)."""
    pr = int(math.isqrt(world))
    while world % pr:
        pr -= 1
    return pr, world // pr


def split(size: int, parts: int, idx: int) -> tuple[int, int]:
    """[start, stop) of part `idx` of `size` items split into `parts` nearly
    equal, contiguous parts."""
    q, r = divmod(size, parts)
    start = idx * q + min(idx, r)
    return start, start + q + (1 if idx < r else 0)


class Grid:
    """The block of C a rank owns and the groups it reduces over."""

    def __init__(self, m: int, n: int, rank: int, world: int, row_group=None, col_group=None):
        self.pr, self.pc = grid_shape(world)
        self.a, self.b = divmod(rank, self.pc)
        self.rows = split(m, self.pr, self.a)
        self.cols = split(n, self.pc, self.b)
        self.row_group, self.col_group = row_group, col_group

    @staticmethod
    def make_groups(world: int, backend=None):
        """Process groups of each grid row and each grid column (every rank
        must call this, in the same order).  Returns (row_groups, col_groups),
        indexed by grid row / grid column."""
        pr, pc = grid_shape(world)
        rows = [dist.new_group([a * pc + b for b in range(pc)], backend=backend) for a in range(pr)]
        cols = [dist.new_group([a * pc + b for a in range(pr)], backend=backend) for b in range(pc)]
        return rows, cols

    @classmethod
    def current(cls, m: int, n: int, backend=None) -> "Grid":
        rank, world = dist.get_rank(), dist.get_world_size()
        rows, cols = cls.make_groups(world, backend)
        g = cls(m, n, rank, world)
        g.row_group, g.col_group = rows[g.a], cols[g.b]
        return g


def reduce_bounds(R: torch.Tensor, K: torch.Tensor, grid: Grid) -> None:
    """In place: R (this block's rows) becomes the maximum over the ranks that
    share the row block, K (this block's columns) over those that share the
    column block.  Skipped when a group has one rank."""
    if grid.pc > 1:
        dist.all_reduce(R, op=dist.ReduceOp.MAX, group=grid.row_group)
    if grid.pr > 1:
        dist.all_reduce(K, op=dist.ReduceOp.MAX, group=grid.col_group)


def gemm_block(A_rows: torch.Tensor, Bt_cols: torch.Tensor, num_moduli: int, mode, grid: Grid,
               out=None, stream=None) -> torch.Tensor:
    """This rank's block C[rows, cols] of A @ B, from A's row block (m_a x k)
    and B's column block given as Bt (n_b x k)."""
    from . import binding as os2
    if os2._mode(mode) == os2.MODE_FAST:
        return os2.gemm(A_rows, Bt_cols, num_moduli, "fast", out=out, stream=stream)
    R, K, EA, EB = os2.scale_bounds(A_rows, Bt_cols, stream=stream)
    reduce_bounds(R, K, grid)
    e = os2.exponents_from_bounds(R, EA, num_moduli, stream=stream)
    f = os2.exponents_from_bounds(K, EB, num_moduli, stream=stream)
    return os2.gemm_exponents(A_rows, Bt_cols, num_moduli, e, f, out=out, stream=stream)
