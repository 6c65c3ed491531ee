"""fp64 CPU oracle of the MoE layer forward -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` leg may
import this package.  It shares no code with the CUDA library in
``expert_routed_ffn_router_gb300``.
"""
from .oracle import (build_oracle, combine, dispatch, expert_rows, forward, layer_tokens,  # noqa: F401
                     layer_tokens_by_expert,
                     num_threads, router, router_ex, set_num_threads)
