"""GB300-native MoE / DeaMoE small-batch decode layer.

The compute path is the C-ABI library ``libmoe_gb300.so`` (hand-written sm_103a
CUDA); :mod:`.binding` marshals torch tensors into its entry points.
"""
