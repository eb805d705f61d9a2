"""GB300-native ForkAttention token-mixing layer.

The compute path is the C-ABI library built from ``csrc/`` (see
``tree_forked_hybrid_gb300.fork`` for the Python binding).  Importing the
package does not load the library; ``workloads`` only draws inputs.
"""
