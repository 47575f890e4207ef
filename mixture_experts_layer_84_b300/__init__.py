"""B300-native (sm_103a) single-GPU MoE layer forward.

The compute path lives in the C-ABI library libmoe.so (include/moe.h); this
package holds its thin Python binding, the workload table and the seeded
synthetic-input generator.
"""
