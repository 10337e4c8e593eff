"""B300-native (sm_103a) draft-tree verification for Gated DeltaNet layers.

The CUDA kernels sit behind a C ABI (``include/gdn_tree.h``, ``libgdn_tree.so``);
``gated_deltanet_tree_03_b300.binding`` is a thin ctypes binding with the same names.
``workloads`` draws the seeded synthetic inputs.
"""

__all__ = ["binding", "workloads"]
