"""fp64 CPU oracle for Stochastic Attention (SA), sliding-window attention (SWA)
and the gated SA+SWA merge.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the ``libsa`` C-ABI
library, its CUDA kernels, or the Python binding) may import, call or link
anything in this package.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.

The oracle is a plain, slow, obviously correct restatement of the method as the
source pages define it ("Stochastic Attention" technical summaries at
gist.science/ja/paper/2604.00754 and gist.science/ko/paper/2604.00754):

* ``prng``      -- splitmix64 and the seeded Fisher-Yates draw of sigma
                  (section "Core mechanism", step 1: sigma ~ Uniform(S_n)).
* ``attention`` -- SA, SWA, the gated dual path and full attention, in fp64,
                  written per ORIGINAL token i over its neighbour set
                  (sections "Core mechanism" steps 1-3, "Theoretical
                  properties" causal bullet, "Gated SA and SWA" equation).
* ``backward``  -- gradients of SA, SWA and the gated merge with respect to
                  Q, K, V and the gate logits, and each row's log-sum-exp
                  (the chain rule through the forward definition; the pages
                  use SA to pretrain a model: "Main contributions", item 3).
* ``prologue``  -- the two gate projections of the layer input and the
                  rotary position embedding by original token index that
                  feed the attention paths ("Gated SA and SWA" section).
* ``graph``     -- neighbour sets, the pairwise connection probability and the
                  receptive-field growth over stacked layers
                  (section "Core mechanism", last paragraph; "Theoretical
                  properties", receptive-field bullet).

It shares no code with the CUDA path; the only module both sides use is
``sa_synth`` (seeded input arrays, no attention arithmetic).
"""

from .prng import splitmix64_step, stream_state, make_perm, inverse_perm
from .attention import (
    sa_rows,
    swa_rows,
    gated_rows,
    sigmoid,
    sa_forward,
    swa_forward,
    gated_forward,
    full_attention,
    masked_attention,
)
from .backward import (
    sa_backward,
    sa_dq_rows,
    swa_backward,
    gated_backward,
    sa_lse,
    swa_lse,
)
from .prologue import gate_logits, rope, rope_angles
from .graph import (
    neighbours_sa,
    neighbours_swa,
    adjacency_sa,
    adjacency_swa,
    pair_probability_closed_form,
    expected_degree_closed_form,
    receptive_field_sizes,
    attended_pairs_closed_form,
)

__all__ = [
    "splitmix64_step",
    "stream_state",
    "make_perm",
    "inverse_perm",
    "sa_rows",
    "swa_rows",
    "gated_rows",
    "sigmoid",
    "sa_forward",
    "swa_forward",
    "gated_forward",
    "full_attention",
    "masked_attention",
    "gate_logits",
    "rope",
    "rope_angles",
    "sa_backward",
    "sa_dq_rows",
    "swa_backward",
    "gated_backward",
    "sa_lse",
    "swa_lse",
    "neighbours_sa",
    "neighbours_swa",
    "adjacency_sa",
    "adjacency_swa",
    "pair_probability_closed_form",
    "expected_degree_closed_form",
    "receptive_field_sizes",
    "attended_pairs_closed_form",
]
