"""CPU oracle for the two fused causal attention forwards (TEST INFRASTRUCTURE).

This package is the slow, plain, obviously-correct definition of what the CUDA
path computes, written in float64 numpy from the source pages:

* ``oracle.tra``   -- threshold rectified attention (TRA), from the page
  "triton_threshold_attention.py" (module docstring formula and the forward
  kernel ``_threshold_rela_fwd_kernel``).
* ``oracle.nsa``   -- NSA selection-branch attention, from the page
  "nsa_selection_kernel.py" (module docstring "The operation" and the
  ground-truth function ``selection_forward_reference``).
* ``oracle.fsa``   -- the same NSA selection forward in the page's block-outer
  split-K form (per-(query, block) softmax partials and a log-sum-exp
  combine), from the page's FSA forward section.
* ``oracle.brute`` -- scalar pure-Python loops of both, for tiny inputs only.

It is test infrastructure.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import it.  It shares no
code with the CUDA library and never imports it; the library never imports
this package.  Every input reaches it as a float64 numpy array (bf16 tensors are
upcast exactly before they arrive).

Parity status: every public function here is pinned by CPU tests against
closed forms, hand-worked fixtures, textbook/library special cases and
invariants (``tests/test_oracle.py``); none is "parity unpinned".
"""

from . import brute, fsa, nsa, tra  # noqa: F401

__all__ = ["tra", "nsa", "fsa", "brute"]
