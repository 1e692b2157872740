"""GB300-native chunked-prefill paged attention step.

The compute path is the C-ABI CUDA library ``libcpa.so`` (sources in
``csrc/``, declared in ``include/cpa.h``); ``ops`` is its thin Python binding.
``sched``, ``batch``, ``workloads`` and ``synth`` are host-side helpers that
compose hybrid batches (decode-first token budget, packed metadata, paged
allocation) and draw seeded synthetic inputs.  Importing the package does not
load the CUDA library; the first call through ``ops`` does, and fails loudly
if it has not been built.
"""
__all__ = ["ops", "sched", "batch", "workloads", "synth"]
