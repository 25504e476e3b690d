"""GB300-native MXFP4 routed-expert MoE feed-forward layer.

The compute path is the C-ABI library ``libmoe_gb300.so`` (CUDA, sm_103a) built
from ``csrc/``; ``binding`` is a thin ctypes layer over it with the same entry
point names (import it explicitly: ``from mxfp4_routed_expert_router_gb300
import binding``).  ``workloads`` holds the seeded synthetic inputs.
"""
