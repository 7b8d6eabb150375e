"""librcc: tensor collectives over R logical ranks on one GB300, plus the
gradient-sync + fused AdamW step that consumes them.

`gradient_sync_rcc_gb300.rcc` is the Python binding of the C ABI declared in
include/rcc.h (argument marshalling only; every step runs in the CUDA
library).  `gradient_sync_rcc_gb300.synth` draws the seeded synthetic inputs.
"""
