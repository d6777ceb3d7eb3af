"""GB300 (sm_103a) DeepSeek sparse-attention decode path.

``libdsa.so`` (built from ``csrc/`` by :mod:`.build`) holds every kernel:
the device-side indexer schedule, the paged lightning-indexer MQA logits
(tcgen05 + TMA), the per-row top-k and the sparse MLA decode.  This package is
the thin Python side: :mod:`._abi` marshals arguments to the C ABI declared in
``include/dsa.h``, :mod:`.step` strings the calls of one decode / prefill step
together over caller-owned buffers, and :mod:`.inputs` draws seeded synthetic
workloads.  There is no CPU or PyTorch fallback: without libdsa.so every call
raises.
"""
__all__ = ["inputs", "step"]
__version__ = "1.0.0"
