"""Float64 CPU oracle for DP-SGD-RC per-sample norm estimation, clipping and noise.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its
Python binding) imports, links or runs anything in this package.  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

The oracle is written from the notes on "Efficient DP-SGD for LLMs with Randomized
Clipping" (ICML 2026, arXiv 2605.24879) and is deliberately plain: float64 numpy,
library matmuls and a library QR as single steps, no blocking, fusion or
reordering beyond what the method's definitions state.  It shares no code with
the CUDA path; only the seeded input generators feed both.

Modules
-------
norms   exact norm (direct, ghost, trace forms), Hutchinson, Hutch++, layerwise
        sum, clip factors.
philox  Philox4x32-10 counter-based generator (Salmon et al., SC'11), the
        uniform -> normal transform and the Gaussian noise add.
rademacher  the +-1 projection variant (signs from the Philox stream, 1/k scale).
cost    the analytic FLOP / memory counts behind the pages' efficiency table.

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (brute force, closed forms, distribution laws,
the pages' printed ratios, or an independent Philox implementation).
"""

from .norms import (  # noqa: F401
    exact_norm,
    ghost_norm,
    trace_norm,
    brute_force_norm,
    hutch_norm,
    hutchpp_norm,
    hutchpp_parts,
    layer_sum,
    clip_factors,
)
from .philox import (  # noqa: F401
    philox4x32_10,
    philox_words,
    normals_from_words,
    noise_normals,
    add_noise,
)
from .rademacher import (  # noqa: F401
    rademacher_signs,
    hutch_norm_rademacher,
    rademacher_variance,
)
from . import cost  # noqa: F401
