"""Plain fp64 CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import or call this
package.  The product path (the CUDA library and its Python binding) never
imports, links or executes anything in here, and this package imports
nothing from the product path.
"""

from .spec_verify_oracle import (  # noqa: F401
    NEAR_TIE,
    SV_GREEDY,
    SV_SAMPLE,
    decode_logits,
    process_row,
    pair_step,
    final_pick,
    pick_admissible,
    topp_sizes,
    row_alternatives,
    admissible_outcomes,
    decide_request,
    conf_label,
    Processed,
    verify_request,
    spec_verify_oracle,
)
from .dspark_schedule_oracle import (  # noqa: F401
    prefix_survival,
    schedule_prefix,
    expected_tokens,
)
