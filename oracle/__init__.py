"""float64 CPU oracle for the HYPIC linear-layer caching path.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or executes
this package; only the tests, ``__graft_entry__.smoke()`` and the bench's CPU
baseline leg do.  It shares no code with the CUDA path: it reads the seeded
inputs (``linear_attn_state_gb300.synth``) and nothing else from the package.

Every function is a plain restatement of what the HYPIC pages define, token by
token, in float64, with each per-token transition formed explicitly:

* ``linear_state``  -- per-token transitions, segment pair (T_C, S(C|0)),
  composition, naive addition, seam-window advance;
* ``schedule``      -- varlen offsets, seam-window body ranges and the
  longest-processing-time-first (LPT) work order.

Parity status: every function here is pinned by the CPU tests (closed forms,
brute force, invariants).  The one number the pages print for this path that
is not fully pinned is the "22% of the state norm" naive-add error: the pages
do not give the model, head or metric, so it is reproduced only by the RetNet
closed form (parity unpinned as a model-level figure).
"""
from . import linear_state, schedule  # noqa: F401
