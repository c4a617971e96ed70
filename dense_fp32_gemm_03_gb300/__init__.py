"""GB300-native FP32 GEMM (C = A * B, row-major, FFMA arithmetic) for sm_103a.

The product is the C-ABI library ``libsgemm.so`` (``include/sgemm.h``); this
package builds it (``_build``), binds it (``binding``) and provides the seeded
synthetic workloads (``workloads``).
"""
from .binding import (AUTO, GUARDED, SMALL, SPECIALIZED, STAGED, STREAMK, STREAMK_SMALL, TILED, TILED_SMALL, VARIANTS,
                      SgemmError, debug_expire_wait, debug_owner_publishes, load, query_device_status,
                      release_workspaces, select_variant, sgemm, sgemm_ex, sgemm_ex2, sgemm_host, sgemm_raw, sgemm_tf32, status_string,
                      ROW_MAJOR, COL_MAJOR, OP_N, OP_T,
                      variant_name, workspace_size)

__all__ = ["sgemm", "sgemm_ex", "sgemm_ex2", "sgemm_host", "ROW_MAJOR", "COL_MAJOR", "OP_N", "OP_T", "sgemm_tf32", "sgemm_raw", "select_variant", "workspace_size", "query_device_status",
           "debug_expire_wait", "debug_owner_publishes", "release_workspaces", "status_string", "variant_name", "load",
           "SgemmError", "VARIANTS", "AUTO", "GUARDED", "TILED", "STREAMK", "TILED_SMALL",
           "STREAMK_SMALL", "STAGED", "SPECIALIZED", "SMALL"]
