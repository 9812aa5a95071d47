"""fp64 CPU oracle (test infrastructure; never on the product path)."""
from .mm_oracle import (  # noqa: F401
    RENORM_EPS, silu, swiglu_ffn, router_logits, softmax, topk, renormalise,
    expert_load, mean_prob, aux_loss_from_stats, aux_loss, combine,
    moe_forward, moe_route, near_tie_tokens, logsumexp, z_loss,
    swiglu_ffn_backward, moe_backward, rms_norm, swiglu_block, moe_block,
)
