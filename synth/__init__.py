"""Seeded synthetic inputs for the FP8 paged MQA-logits indexer.

This module only draws random numbers and packs them into the byte layouts the
indexer consumes. It holds none of the indexer's arithmetic, and both the CPU
oracle and the CUDA path take their inputs from here.
"""

from .inputs import (  # noqa: F401
    CONFIGS,
    PREFILL_CONFIGS,
    PrefillProblem,
    Problem,
    config_problem,
    make_prefill,
    make_problem,
    pack_kv,
    prefill_config,
    prefill_ranges,
)
