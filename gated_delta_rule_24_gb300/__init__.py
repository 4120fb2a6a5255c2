"""GB300-native chunked Gated Delta Rule (GDN) prefill.

The compute path is a C-ABI CUDA library (``csrc/``, built for sm_103a, C ABI
in ``include/gdn.h``); this package holds its thin Python binding and the
seeded workload generators.  The binding loads the library on first use and
fails loudly when it is missing: there is no CPU fallback.
"""
from .binding import (GdnError, chunk_gated_delta_rule, device_status, gdn_chunk_prefill,  # noqa: F401
                      gdn_chunk_prefill_checkpointed, gdn_chunk_prefill_noalloc,
                      gdn_decode_step, gdn_init, gdn_reserve_workspace, gdn_split_workspace_bytes,
                      load_library, run_problem, testing_force_splits, testing_split_plan,
                      testing_wait_limit)
