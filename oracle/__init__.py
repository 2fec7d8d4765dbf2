"""CPU oracle for the Kimi Delta Attention (KDA) recurrence.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import this package. The
CUDA library never calls it and shares no code with it; the two meet only in
the seeded input generators, which hold none of the method's arithmetic.

Three independent restatements of the same definition (Kimi K3 -- Architecture
Notes, section 1.1 "Kimi Delta Attention"):

* ``recurrent`` -- the defining token-by-token recurrence in plain C, fp64
  (``kda_oracle.c``), threaded over (sequence, head) pairs. This is the oracle
  the GPU path is compared with. ``kda_recurrent_gated`` is the same recurrence
  with the log-decay of the gated form, ``g = g_min * Sigmoid(e^{A_h} z)``
  (section 1.2, the K3 row of the mapping table); ``kda_recurrent_unbounded``
  the unbounded map of the earlier models, ``g = -e^{A_h} Softplus(z)``.
* ``chunked``  -- the chunkwise form (section 1.2: "recurrent across chunks and
  parallel within each chunk") in numpy fp64, with the chunk's triangular
  system solved by a library inverse. Pinned to ``recurrent`` by agreement.
* ``exact``    -- the recurrence with explicit dense transition matrices in
  exact rational arithmetic (``fractions.Fraction``), for tiny inputs.
* ``epilogue`` -- the output gate with head-wise RMSNorm of section 1.3
  ("Full-rank output gate"), applied to a read-out, in numpy fp64.
* ``prologue`` -- the input prologue of section 1.1 (short convolution, Swish,
  L2 norm of q and k), with per-sequence convolution states, in numpy fp64.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(exact brute force, closed forms, invariants, recurrent/chunked agreement and
planted-mistake checks). No worked numeric example exists on the pages, so no
pin is a printed value.
"""

from .recurrent import (kda_recurrent, kda_recurrent_mutant, kda_recurrent_gated, MUTATIONS,  # noqa: F401
                        GATE_MUTATIONS, oracle_library_path, kda_recurrent_unbounded, UNBOUNDED_MUTATIONS)
from .chunked import kda_chunked, chunk_quantities  # noqa: F401
from .exact import kda_exact  # noqa: F401
from .epilogue import output_gate_rmsnorm, EPILOGUE_MUTATIONS  # noqa: F401
from .prologue import kda_prologue, short_conv, PROLOGUE_MUTATIONS  # noqa: F401
