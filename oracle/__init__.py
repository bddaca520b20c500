"""fp64 CPU oracle of one nanochat-style GPT training step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it.  It shares no code with the CUDA path.

The model it computes is the one the nanochat pages describe:

* cosmicrealm "noao-chat-0-项目总体介绍" §2.1 items 1-6: half-split RoPE, QK
  norm after RoPE, untied embedding / lm_head, relu² MLP, parameter-free
  RMSNorm with bias-free linears, grouped-query attention;
* devpress "用不到100美元，亲手训练一个属于你的GPT-2" §4.1: decoder block with
  normalisation, causal self-attention and a feed-forward net; §4.2: fp32
  master weights cast to the compute dtype in the forward;
* woshipm nanochat analysis §五.1: a 4x feed-forward layer.

``optim.py`` restates the optimizer step that follows the gradients (Muon for
the weight matrices, AdamW for the embedding and the output head;
cosmicrealm §2.2 and §4.2).

Readings taken where the pages are silent are listed in each function's
docstring.  Parity of the whole step is pinned by finite differences and by the
invariants in ``tests/test_oracle_*.py``.
"""
from .rng import splitmix64_outputs, normal_init, init_params
from .model import (Config, param_layout, n_params, rms_norm, rms_norm_bwd,
                    rope_tables, rope, rope_bwd, attention, attention_bwd,
                    cross_entropy, softcap, forward_logits, forward_backward,
                    row_losses, unpack, pack)
