"""CPU oracle of the MoL LoRA hot path -- test infrastructure only.

Imported by the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline and reference arm; never by the product path.
"""

from .mol_oracle import *  # noqa: F401,F403
from .mol_oracle import (  # noqa: F401
    bf16_to_f64, f64_to_bf16, virtual_topk, align_capacity, align_block_size,
    lora_shrink, lora_expand, lora_forward_stage, brute_force_stage, token_lora_ids, MAX_BUCKETS,
)
