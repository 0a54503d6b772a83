"""Host-side check of the full-size GPU parity tests' row sampling: the
sampled rows reach every (rank, shard, 128-row block) of every AllGather->GEMM
task and every (bucket, 128-row block) of every GEMM->ReduceScatter bucket of
the MLP sweep, so every CTA half of every pair tile is compared with the
oracle at every N and chunk count."""

import numpy as np

from collective_matmul_decomposition_gb300 import inputs as gen
from test_gpu_parity import BLOCK, _ag_rows, _rs_rows


def test_sample_rows_cover_every_task_and_block():
    """The sampled rows reach every (rank, shard, 128-row block) and every
    (bucket, 128-row block) of the MLP sweep at every N."""
    rng = np.random.default_rng(0)
    for N in (4, 8, 16):
        s = gen.mlp_shapes(N)
        m, Mb = s["ag"]["m"], s["rs"]["M"] // N
        ranks, rows = _ag_rows(N, m, rng)
        got = {(int(r), int(i) // m, (int(i) % m) // BLOCK) for r, i in zip(ranks, rows)}
        assert got == {(r, j, b) for r in range(N) for j in range(N) for b in range(m // BLOCK)}
        owners, orow = _rs_rows(N, Mb, rng)
        got = {(int(o), int(i) // BLOCK) for o, i in zip(owners, orow)}
        assert got == {(o, b) for o in range(N) for b in range(Mb // BLOCK)}
