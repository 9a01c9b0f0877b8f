"""CPU fp64 oracle (test infrastructure only; see seg_attn.py, seg_paged.py)."""
from .seg_paged import brute_force_paged, gather_head, seg_paged_request
from .seg_attn import (attend, attend_partial, bitmap_words, brute_force, build_protected,
                       lse_merge, relocate, restore_output_phase, rope_theta, rotate,
                       seg_attn_request, visible_keys)

__all__ = ["brute_force_paged", "gather_head", "seg_paged_request", "attend", "attend_partial", "bitmap_words", "brute_force", "build_protected",
           "lse_merge", "relocate", "restore_output_phase", "rope_theta", "rotate", "seg_attn_request", "visible_keys"]
