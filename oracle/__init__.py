"""Plain fp64 CPU oracle for the Megatron tensor-parallel Transformer block.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never calls it and
shares no code with it: no kernels, helpers, constants or table generators.

What it computes is the *unsharded* definition of each block, written out in
numpy float64 with library matmuls as the only primitive, so that a reader can
check it against the pages by eye.  Separate ``*_sharded`` routines compute the
same block as n per-rank partials summed afterwards; they exist to pin the
unsharded routines to the pages' sharding identities.

Pages cited (short name -> page title):

* [Grasp-TP]  Grasp lesson 11, "张量并行线性层分片与前反向通信量计算"
  (tensor-parallel linear-layer sharding and forward/backward communication).
* [Troverld]  cnblogs post "ラブパラ" by Troverld, a survey of parallelisms
  (sections O.I Notation, O.II Collective Communication, I.III Tensor
  Parallelism, II.II Communication Approaches, II.III Computational Details).
* [hjcheng-TP] hjcheng0602 blog post "TP" (sections MLP / Attention,
  单卡forward, 单卡backward, TP forward, TP backward).
* [adu-TP]    "Tensor Parallelism张量并行（一）", notes on the Megatron-LM paper
  (sections 行切分, 列切分, 张量并行应用于 MLP 和 Attention, 算子 f 和 g,
  张量并行的通信开销).

Parity status of each function is stated in its docstring; the only unpinned
item is the worked communication example of [Grasp-TP] §5, whose numbers were
lost from the page, so nothing here reproduces it.
"""

from .primitives import (gelu, gelu_grad, silu, silu_grad, sigmoid,
                         splitmix64_mix, splitmix64_stream, dropout_threshold,
                         dropout_keep)
from .mlp import (mlp_forward, mlp_backward, mlp_forward_sharded,
                  mlp_backward_sharded)
from .attention import (attention_forward, attention_backward,
                        attention_forward_sharded, attention_backward_sharded)
from .norm import rmsnorm_forward, rmsnorm_backward
from .layer import layer_forward, layer_backward
from .accounting import (comm_report, mlp_flops, attn_flops, layer_flops,
                         act_memory)
from . import sampled

__all__ = [
    "gelu", "gelu_grad", "silu", "silu_grad", "sigmoid", "splitmix64_mix",
    "splitmix64_stream", "dropout_threshold", "dropout_keep", "mlp_forward",
    "mlp_backward", "mlp_forward_sharded", "mlp_backward_sharded",
    "attention_forward", "attention_backward", "attention_forward_sharded",
    "attention_backward_sharded", "rmsnorm_forward", "rmsnorm_backward",
    "layer_forward", "layer_backward", "comm_report", "mlp_flops",
    "attn_flops", "layer_flops", "act_memory", "sampled",
]
