"""activation_backward_gb300 -- the backward pass of a darknet/caffe-style
convolutional layer (activation gradient, batch-norm backward, bias/scale
updates, weight gradient, input gradient with the shortcut delta) as
hand-written CUDA for GB300 (sm_103a), behind a C ABI (``include/cba.h``).

``_binding`` is the ctypes binding (same names as the C ABI); ``layer`` holds
the device-side convenience wrapper; ``inputs`` generates seeded synthetic
workloads.  The CUDA library is loaded lazily; nothing falls back to the CPU.
"""
from ._binding import (ACT_NAMES, CBA_ACT_ELU, CBA_ACT_HARDTAN, CBA_ACT_LEAKY,  # noqa: F401
                       CBA_ACT_LHTAN, CBA_ACT_LINEAR, CBA_ACT_LOGGY, CBA_ACT_LOGISTIC,
                       CBA_ACT_PLSE, CBA_ACT_RAMP, CBA_ACT_RELIE, CBA_ACT_RELU, CBA_ACT_SELU,
                       CBA_ACT_STAIR, CBA_ACT_TANH, CBA_ERR_ALIGN, CBA_ERR_ARG,
                       CBA_ERR_CUDA, CBA_ERR_DEVICE_TIMEOUT, CBA_ERR_SCRATCH_LIMIT,
                       CBA_ERR_UNSUPPORTED, CBA_ERR_WORKSPACE, CBA_MATH_FFMA, CBA_MATH_TF32,
                       CBA_NOALLOC_MAX_K, CBA_OK, CbaError, cba_bn_act_backward_noalloc,
                       cba_conv_bn_act_backward, cba_conv_bn_act_backward_traced, cba_desc_t,
                       cba_error_string, cba_get_status, cba_last_cuda_error,
                       cba_selftest_bounded_wait, cba_version, cba_workspace_bytes, load,
                       make_desc, CBA_ROUTE_MAX_INPUTS, cba_maxpool_backward,
                       cba_pool_desc_t, cba_pooled_size, cba_route_backward, cba_yolo_backward,
                       make_pool_desc, CBA_WS_RECOMPUTE_Z, cba_workspace_bytes_ex,
                       cba_conv_bn_act_backward_grouped, cba_workspace_bytes_grouped,
                       cba_plan_info, CBA_PHASE_EVENTS, CBA_PATH_FFMA, CBA_PATH_TC_ROWS,
                       CBA_PATH_TC_BATCH_INNER, CBA_PATH_TC_GEMM_1X1)
