"""GB300-native batch-1 Qwen-style decode step behind the qw_* C ABI (include/qw.h).

``_binding`` is the ctypes layer over libqw.so (same names as the header);
``device_model.DeviceModel`` uploads a drawn workload and drives a handle;
``build_lib.build()`` compiles the sm_103a library in-tree.
"""
from . import _binding  # noqa: F401
from ._binding import (  # noqa: F401
    QwError, lib, qw_create, qw_decode_greedy, qw_decode_step, qw_destroy, qw_get_capture,
    qw_get_pos, qw_kv_cache, qw_load_weights, qw_prefill, qw_reset, qw_set_capture,
    qw_set_lora, qw_set_pos, qw_set_wait_limit_ns,
)
