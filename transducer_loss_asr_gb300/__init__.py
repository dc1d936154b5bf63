"""GB300-native (sm_103a) Token-and-Duration Transducer (TDT) loss.

The loss and its gradient run in one call of the C ABI declared in
``include/tdt_loss.h`` and implemented by ``libtdt_loss.so`` (CUDA kernels
under ``csrc/``).  ``binding`` marshals PyTorch tensors into that ABI;
``workloads`` makes the seeded synthetic inputs.  Importing this package does
not load the library; ``from transducer_loss_asr_gb300 import binding`` does,
and raises if it has not been built.
"""

__all__ = ["binding", "workloads", "build"]
