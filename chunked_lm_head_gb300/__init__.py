"""libflce: chunked fused LM-head cross-entropy on GB300 (sm_103a).

The compute lives in the C-ABI CUDA library (include/flce.h, csrc/); this
package holds its ctypes binding, a thin torch-facing API and the seeded
synthetic workloads.
"""
from .api import (IGNORE_INDEX, DistillLoss, GRPOLoss, LinearCrossEntropy,  # noqa: F401
                  LinearCrossEntropyLoss, SelectiveLogSoftmax,
                  backward, distill_loss, forward, forward_backward, grpo_loss, grpo_token_loss,
                  jsd_backward, jsd_forward, kd_backward, kd_forward, linear_cross_entropy,
                  scale_grads, selective_log_softmax, workspace_bytes)
