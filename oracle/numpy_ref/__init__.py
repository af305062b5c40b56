"""Independent float64 numpy restatement of the oracle's definitions (test
infrastructure, not product).

The oracle itself is the C++ library of the parent package. This numpy
version (BLAS products, vectorised) computes the same definitions in a second,
independent way; ``tests/test_oracle_cross.py`` checks that the two agree.
Nothing else uses it. Only ``tests/`` may import it."""
from .gate import (cosine_similarity, cosine_gate, router_probability, router_gate,
                   earliest_exit, layer_ops)  # noqa: F401
from .compact import stable_partition, gather_rows, exit_scatter  # noqa: F401
from .fill import dequant_int4, rms_norm, rope_rotate_half, fill_rows, kv_fill  # noqa: F401
from .ridge import ridge_fit  # noqa: F401
from .river import silu, attention, exit_layer, exit_river  # noqa: F401
