"""GB300-native (sm_103a) DSpark ragged-verification hot path.

Four calls make one decode step of confidence-driven variable-length speculative
verification ("DSpark in SGLang: Speculative Decoding with Confidence-Driven, Variable-Length
Verification"): dspark_schedule -> dspark_pack -> dspark_verify -> dspark_scatter. They are
implemented as hand-written CUDA kernels in libdspark.so (C ABI: include/dspark.h); this
package is the ctypes binding (`_binding`), the in-tree build (`build`), a buffer-owning step
runner (`step`) and the seeded synthetic workloads (`synth`).
"""
from ._binding import (BF16, CAP_ACCEPT, COMPACT, F32, MODES, STATIC, CostTable, DSparkError,  # noqa: F401
                       dspark_pack, dspark_scatter, dspark_schedule, dspark_verify,
                       dspark_verify_workspace_bytes, last_error, lib, version)
