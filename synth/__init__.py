"""Seeded synthetic inputs for the FP8 paged MQA-logits indexer and the
sparse MLA decode that consumes its top-k positions.

This module only draws random numbers and packs them into the byte layouts the
indexer and the decode consume. It holds none of their arithmetic, and both the CPU
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
from .mla import MLA_CONFIGS, MlaProblem, make_mla_problem, mla_config  # noqa: F401,E402
