"""GB300 (sm_103a) W4 MoE expert layer: GPU-resident routing, fused-dequant
tcgen05 grouped GEMMs and a W4 GEMV decode path behind a C ABI
(include/lily_moe.h).  This package is the thin Python binding; the compute
runs in liblily_moe.so, built by ``build.build()``."""
from ._lib import *  # noqa: F401,F403
from ._lib import (Dims, LayerWeights, RoutingBuffers, LilyError, alloc_workspace, make_dims,
                   lib, EXPORTS, LIB_PATH)  # noqa: F401
