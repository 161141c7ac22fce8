"""fp64 CPU oracle for the generalised gated delta-rule recurrence.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import, call or execute anything in this
package.  The product (the C-ABI library and its Python binding) never routes
through it, and it shares no code, table or helper with the CUDA path: the
only thing both sides consume is the seeded input generator module, which
holds none of the method's arithmetic.

Modules
-------
recurrence  Tokenwise recurrence (the plain definition) for GDN, KLA, PGDN,
            Diagonal KDN, KDA, PKDA, isotropic KDN and the exact Kalman memory
            (dense key covariance), one token at a time, in float64.
chunkwise   A naive chunkwise-parallel restatement (triangular system per
            chunk), written independently of ``recurrence`` as a cross-check.
backward    Reverse-mode gradients of the tokenwise recurrence (every variant)
            w.r.t. q, k, v, log-decay, every gate,
            the initial state and the gain state's initial value; and the same
            gradients through the chunkwise form (every chunkwise variant).
ridge       Side oracles fixed by closed forms: exact ridge regression (ATQ),
            its Sherman-Morrison recursion (ATK), the diagonal counterexample
            and a dense-covariance Kalman filter.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against values printed on the pages, closed forms, library routines or
brute force; none is "parity unpinned".
"""

from .recurrence import (  # noqa: F401
    VARIANTS,
    TOKENWISE_ONLY,
    l2normalize,
    gdn_write,
    kla_write,
    pgdn_stat_update,
    pgdn_squash,
    kdn_predict,
    kdn_gain,
    kdn_variance_update,
    ikdn_predict,
    ikdn_gain,
    ikdn_variance_update,
    ekdn_predict,
    ekdn_gain,
    ekdn_cov_update,
    recurrence_step,
    tokenwise,
)
from .chunkwise import chunkwise, pgdn_stat_chunk, kdn_mobius_chunk  # noqa: F401
