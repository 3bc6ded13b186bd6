"""CPU oracle for the affinity-aware MoE layer forward -- TEST INFRASTRUCTURE.

Plain, slow, obviously-correct numpy (float64) restatement of what the layer
computes, used only by the tests, by the package's smoke check and by the
benchmark's CPU-baseline leg.  The product path never imports it and shares no
code with it: no kernels, headers, helpers or tables.

Sources (the pages' titles and sections):

* Semantic Parallelism: Redefining Efficient MoE Inference via Model-Data
  Co-Scheduling -- the Korean (ko), German (de) and Japanese (ja) summaries.
  Token-expert affinity and the token-id lookup table (ja §2.1, §2.3;
  de §2 A), the local activation rate (ko §3, de §4), and the
  Shuffled-Reduce-Scatter / Shuffled-Allgather shuffle pair that moves tokens
  to the rank hosting their experts and restores their order (ko §2.2,
  de §2 B, ja §2.2 B).
* MoE-Prism: Disentangling Monolithic Experts for Elastic MoE Services via
  Model-System Co-Designs (ko) -- per-request routing budget k (§1, §2 B, §5)
  and sub-experts (§2 A).

The pages fix no router maths and no expert-FFN form.  The readings taken are
stated in each function's docstring (fp32 softmax; top-k by descending logit
with ties to the lowest expert index; gates renormalised over the selected
experts; SwiGLU experts).

Parity is pinned by the CPU tests (brute force, invariants, closed forms and a
hand-derived worked example); nothing here is unpinned.
"""
from .moe import (  # noqa: F401
    round_to, bf16_round, silu, router_logits, topk_route, affinity_lookup,
    remote_count, physical_order, permute, expert_ffn, grouped_ffn, shared_ffn, combine,
    moe_layer,
)
from .scheduling import dp_schedule, transition_lookup  # noqa: F401
from .prism import hier_route, split_expert_weights, sub_scores  # noqa: F401
