"""B300 (sm_103a) DyRA linear layer: Y ~= X W_hat + b + L R with a per-sample one-step ALS
correction, behind a C ABI (include/dyra.h) and this thin ctypes binding."""
from .dyra import (DyraError, Layer, fit, linear_forward, linear_forward_host,  # noqa: F401
                   linear_forward_profiled, linear_forward_static, load, mlp_forward, new_workspace,
                   prepare, selftest_bounded_wait, workspace_status, workspace_view)
