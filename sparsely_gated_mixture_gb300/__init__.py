"""Sparsely-gated Mixture-of-Experts layer forward path for one GB300 (sm_103a).

The computation runs in hand-written CUDA kernels inside ``libmoe.so``; the
``binding`` module exposes its C-ABI entry points under the same names
(``moe_gate``, ``moe_dispatch``, ``moe_expert_ffn``, ``moe_combine``,
``moe_aux_loss``, ``moe_forward``). Importing this package does not load the
library; the first call into ``binding`` does, and raises if it is missing.
"""
__version__ = "0.1.0"
