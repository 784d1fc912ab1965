"""DSpark per-round speculative-decoding hot path on GB300 (sm_103a).

Markov-head draft -> confidence scheduler -> exact verification, as CUDA kernels behind
the C ABI declared in ``include/dspark.h``.  ``binding`` marshals PyTorch tensors to that
ABI; ``workloads`` generates the seeded synthetic inputs.
"""
from . import workloads  # noqa: F401

__all__ = ["binding", "workloads", "build"]
