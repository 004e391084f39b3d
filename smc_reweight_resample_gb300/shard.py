"""Partition of the SMC-SD step over several GPUs, one process per GPU.

Prompt groups are independent ("Faster LLM Inference via Sequential Monte Carlo", sec. 2: the
effective sample size and the resampling of a prompt concern its own N particles; sec. 3: the
page-table remap moves metadata within those particles). So a job of G groups splits into
contiguous blocks of whole groups, one block per rank; each rank calls smc_step on its block with
its own page-table rows, and the data path needs no collective. The split below gives the first
G % world ranks one group more than the others.
"""
from __future__ import annotations


def group_range(G: int, world: int, rank: int) -> tuple[int, int]:
    """Groups [g0, g1) of rank `rank` among `world` ranks."""
    if G < 0 or world <= 0 or not 0 <= rank < world:
        raise ValueError("need G >= 0, world > 0 and 0 <= rank < world")
    base, extra = divmod(G, world)
    g0 = rank * base + min(rank, extra)
    return g0, g0 + base + (1 if rank < extra else 0)


def particle_range(G: int, N: int, world: int, rank: int) -> tuple[int, int]:
    """Particles [s0, s1) of rank `rank`: the particles of its groups."""
    g0, g1 = group_range(G, world, rank)
    return g0 * N, g1 * N
