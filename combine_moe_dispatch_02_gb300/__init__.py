"""GB300-native MoE token dispatch / combine (one GPU, virtual EP ranks).

The compute path is the CUDA library ``libmoe_ep.so`` (C-ABI declared in
``include/moe_ep.h``); :mod:`combine_moe_dispatch_02_gb300.ep` is its thin
ctypes binding.  :mod:`combine_moe_dispatch_02_gb300.inputs` draws the
seeded synthetic workloads.  Nothing is imported eagerly so that the input
generators work on machines without the CUDA library.
"""
__all__ = ["ep", "inputs"]
