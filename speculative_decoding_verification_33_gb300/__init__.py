"""GB300-native batched speculative-sampling verify step.

The hot path is one CUDA library (``_build/libspecverify.so``, sources in ``csrc/``, C ABI in
``include/spec_verify.h``); ``api`` is its thin torch binding and ``workloads`` makes the seeded
synthetic inputs.
"""
from .api import (device_error, draft_sample, hbm_read_probe, lmhead_stats, residual_topf,
                  spec_verify, to_device_logits, verify, verify_hidden, verify_host)

__all__ = ["spec_verify", "verify", "verify_host", "draft_sample", "residual_topf",
           "lmhead_stats", "verify_hidden", "device_error", "hbm_read_probe",
           "to_device_logits"]
