"""GB300-native paged sparse/sliding-window MQA decode attention.

The compute path is the C-ABI library ``libdsa_decode.so`` (hand-written
sm_103a CUDA kernels, see ``csrc/``); ``binding`` marshals torch tensors into
it. ``workloads`` draws seeded synthetic inputs.
"""
__all__ = ["binding", "workloads"]
