"""B300-native (sm_103a) forward pass of one token-choice MoE FFN layer.

The compute path is the C-ABI library built from csrc/ (libmoe.so); the
`binding` submodule marshals torch tensors into its entry points. `inputs`
draws the seeded synthetic workloads. Import the submodules explicitly.
"""
