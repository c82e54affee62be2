"""CPU oracle for the block-diffusion speculative verification pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the C-ABI library,
its Python binding) imports, links or runs this package; only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may use it.  It shares no code with the CUDA path.

What it computes, plainly and slowly, in float64 (numpy):

* ``mask.verify_mask``        dense allowed-key matrix of one sequence, written
                              out from the temporal attention rule
                              (SimSD summary, section 2 "Temporal Attention Mask").
* ``rope.rope_positions`` /
  ``rope.rotate``             rotary embedding with the RoPE-copy index
                              (SimSD summary, section 3 "Position Encoding Alignment").
* ``attention.verify_attention``  masked softmax attention, one (sequence, head)
                              at a time (SimSD summary, section 4 "Verification").
* ``accept.accept_batch``     acceptance in temporal order: greedy state
                              equality, coupled Gumbel-noise match and standard
                              rejection sampling, longest accepted prefix
                              (SimSD summary section 4 "Acceptance"; SPOT review,
                              section "How it is used").
* ``commit.commit_batch``     the pass's commit into the KV cache: fresh prompt
                              rows, then the accepted data rows in stage order
                              (SimSD summary section 4 "Acceptance", the longest
                              accepted prefix is committed; reading for the layout).
* ``lmhead.accept_lmhead``    the LM head over the mask slots (l = W h, exact,
                              rounded once to fp32) followed by the acceptance
                              above (SimSD summary section 4; SPOT review).

Pins (``tests/test_oracle_*.py``, marked ``not gpu``) tie each function to
something other than itself: a hand-worked mask from the rule's text, mask
counting invariants, the reduction to textbook causal attention for B=1 and
for the identity stage map, the block-state reduction of each mask row to
unmasked attention, the no-leak perturbation property, permutation
equivariance, RoPE's complex-exponential form and relative-position
invariance, brute-force laws of the Gumbel-max and rejection samplers.
The attention *values* at full size carry no printed example on the pages
and rest on those reductions.
"""
from . import mask, rope, attention, accept, commit, lmhead  # noqa: F401
