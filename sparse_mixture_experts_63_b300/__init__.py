"""Single-GPU (B300, sm_103a) forward pass of one sparse Mixture-of-Experts layer.

The compute lives in the C-ABI library ``libmoe.so`` (sources in ``csrc/``,
declarations in ``include/moe.h``).  The functions re-exported here are the
thin ctypes binding to it (``binding``), under the C entry points' names, and
the expert-parallel layer (``expert_parallel``) that drives its kernels around
torch.distributed all-to-all exchanges.
"""
from .configs import CONFIGS, MoEConfig  # noqa: F401
from .binding import (  # noqa: F401
    MoEError, MoELayer, make_forward_args, moe_capacity, moe_combine, moe_expert_ffn,
    moe_forward, moe_forward_host_io, moe_forward_workspace_size, moe_permute,
    moe_ep_regroup, moe_ep_return, moe_router_topk, moe_version)
from .expert_parallel import ExpertParallelMoE, TorchDistExchange  # noqa: F401
