"""CPU oracle for the REINFORCE Zero logprob + importance-sampled loss path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only the test suite, the smoke check and the CPU
baseline leg of the benchmark use it.  It shares no code with the CUDA
library (no kernels, headers, helpers or constant tables) and does not
import it.

Everything is computed in float64 from the exact values of the (bf16)
inputs, step by step in the order the pages define it.  Library
primitives (numpy matmul, exp, log) serve as single steps.
"""

from .rz_oracle import (  # noqa: F401
    lmhead_logits,
    logsumexp_rows,
    token_logprob,
    token_logprob_rows,
    group_advantage,
    is_loss,
    d3,
    loss_fwd_bwd,
    sc_loss,
    sc_loss_fwd_bwd,
    logits_loss_fwd_bwd,
    is_stats,
    peak_to_median,
)
