"""fp64 CPU oracle for the exact attention forward pass (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this
package.  The product path (the CUDA library and its binding) never does.
"""
from .attn_ref import attention, backward, build, num_threads, probabilities

__all__ = ["attention", "backward", "build", "num_threads", "probabilities"]
