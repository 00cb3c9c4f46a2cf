"""GB300 (sm_103a) tile-granular fused GEMM + collective kernels of tensor parallelism.

``gemm_tile_level_gb300.mk``    -- ctypes binding of libmk.so (the C ABI in include/mk.h)
``gemm_tile_level_gb300.api``   -- torch-tensor helpers: device buffers, workspace, calls
``gemm_tile_level_gb300.build`` -- compiles libmk.so in-tree for sm_103a
The binding is imported lazily so that ``build`` works before the library exists; importing
``mk`` or ``api`` without a built libmk.so raises ImportError.
"""
