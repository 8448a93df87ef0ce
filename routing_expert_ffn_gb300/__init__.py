"""Routed-expert path of a Mixture-of-Experts layer, native to GB300 (sm_103a).

libmoe.so (CUDA kernels behind a C ABI, include/moe.h) does the work;
``routing_expert_ffn_gb300.moe`` is its thin Python binding and
``routing_expert_ffn_gb300.inputs`` draws the seeded synthetic workloads.
"""
