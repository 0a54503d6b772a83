"""Decomposed collective matmul (AllGather->GEMM, GEMM->ReduceScatter) on one GB300.

N logical ranks share one GPU's HBM; the ring schedules, the partial GEMMs,
the shard forwarding and the circulating accumulators all run in the CUDA
library behind include/cm.h.  This package is its Python binding.
"""

from .cm import (CMError, Plan, cm_ag_gemm, cm_backward_pair, cm_cannon_gemm, cm_check_status,  # noqa: F401
                 cm_gemm_rs,
                 cm_gemm_rs_pipelined, cost_estimate, load, plan_choose, version)
