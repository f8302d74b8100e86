"""GB300 decode megakernel: one persistent sm_103a kernel per decode step.

The compute path lives in libmk.so (C ABI in include/mk.h); this package holds
its ctypes binding (``_lib``), a tensor-marshalling ``Decoder`` object and the
in-tree build script."""
from ._lib import (MK_ABL_GRAPH, MK_ABL_PDL, MK_ABL_STREAM, MK_ERR_CUDA, MK_ERR_DEVICE,  # noqa
                   MK_ERR_INVALID_ARG, MK_ERR_NOT_READY, MK_ERR_SCHEDULE, MK_ERR_TIMEOUT,
                   MK_ERR_SCRATCH, MK_ERR_UNSUPPORTED, MK_OK, MK_WEIGHTS_BF16, MK_WEIGHTS_INT8, MkError,
                   lib, lib_path, mk_build_schedule, mk_create, mk_create_ex, mk_quantize_rows_int8, mk_debug_drop_instruction, mk_get_routes, mk_decode_step, mk_decode_steps,
                   mk_decode_step_ablation, mk_decode_step_host, mk_decode_step_noalloc, mk_destroy, mk_get_info,
                   mk_plan, mk_plan_check, mk_set_wait_timeout, mk_set_trace, mk_get_trace, mk_set_l2_prefetch, mk_set_residual_copies, mk_set_hold_policy, mk_status_string,
                   mk_sync_status)
from .decoder import Decoder, desc_from_config  # noqa: F401
