"""Full-size parity: the fp64 oracle over row chunks on host threads.

The GPU tier compares every element of the full-size workloads with the
oracle. Computing the oracle for all rows at once would hold several fp64
copies of a 134M-element tensor; instead the rows are cut into chunks, each
chunk runs through the oracle (whose ctypes calls release the GIL, so chunks
run in parallel) and is compared with the matching rows of the GPU result at
once. Peak host memory is a few chunks' worth.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import torch

CHUNK_ROWS = 1024


def host_threads(cap=8):
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(cap, n))


def chunk_rows(H):
    """Rows per chunk: about 8M elements (2048 rows of 4096 features)."""
    return max(CHUNK_ROWS, (1 << 23) // max(1, H))


def row_chunks(M, chunk=CHUNK_ROWS):
    return [(a, min(M, a + chunk)) for a in range(0, M, chunk)]


def for_row_chunks(M, work, chunk=CHUNK_ROWS):
    """Run work(a, b) for every row chunk [a, b) on host threads; the first
    failure (an AssertionError from a comparison) is raised."""
    threads = host_threads()
    prev = torch.get_num_threads()
    torch.set_num_threads(max(1, prev // threads))
    try:
        with ThreadPoolExecutor(max_workers=threads) as pool:
            futs = [pool.submit(work, a, b) for a, b in row_chunks(M, chunk)]
            for f in futs:
                f.result()
    finally:
        torch.set_num_threads(prev)


def rows_of(inp, a, b):
    """Rows [a, b) of every [M, H] input (a view of contiguous rows); the
    weight and other flat tensors whole."""
    return {k: (v[a:b] if v.dim() == 2 else v) for k, v in inp.items()}
