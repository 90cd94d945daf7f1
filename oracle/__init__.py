"""fp64 CPU oracle for the MIS hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
legs may import this package; the product library never does.
"""
from .mis_oracle import *  # noqa: F401,F403
from .mis_oracle import (EMPTY, FULL, PARTIAL, Layout, attention, build_layout,  # noqa: F401
                         CachedLayout, attention_cached, cached_layout, tile_map_cached,  # noqa: F401
                         causal_layout, cost_ratio, label_scores, mask_bruteforce,
                         mask_rows, pair_count, rope, setwise_layout, SetwiseLayout, tile_map,
                         useful_attention_flops)
