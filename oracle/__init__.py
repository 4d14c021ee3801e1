"""fp64 CPU oracle of the K-FAC preconditioning step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything in this package.
The product path (``infra_fac_factors_gb300``) never imports it, and this
package never imports the product path: the two share no code.

Every function is a plain, slow, obviously-correct restatement of the step as
"Accelerating Distributed K-FAC with Smart Parallelism of Computing and
Communication Tasks" (the SPD-KFAC paper) defines it, in float64.  Where the
extracted pages lost a formula or leave a step open, the reading taken is
written next to the function.  Parity status: every function here is pinned by
``tests/test_oracle.py`` (no function is "parity unpinned").
"""
from .kfac import (  # noqa: F401
    factor, shard_factors, aggregate, update_running, damp,
    cholesky_lower, lower_tri_inverse, spd_inverse, damped_inverse,
    precondition, spatial_sum, factor_tile_units, upper_tiles,
    packed_index, kron_precondition_bruteforce, kfac_step, weight_step, stored_part,
    im2col3x3, pack_upper, unpack_upper,
)
