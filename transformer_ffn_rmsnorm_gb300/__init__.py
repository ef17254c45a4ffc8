"""GB300 (sm_103a) pre-norm SwiGLU feed-forward block.

``ffn`` is the Python front end of the C ABI in ``include/ffn.h``; the
computation runs in the hand-written CUDA kernels of ``libffn_gb300.so``
(built by ``build.build()``).  Importing ``ffn`` loads the library and fails
if it is missing.
"""

__all__ = ["ffn", "build"]
