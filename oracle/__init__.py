"""fp64 CPU oracle of the expert-cache MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path never does: it runs entirely in the CUDA library and fails loudly when
that library is missing.  The oracle shares no code with the CUDA path; the
two meet only in the seeded inputs of ``synth``.

Sources, cited by page title and section:

* [Review]  "论文综述：FreeToken 让个人电脑跑起前沿 MoE 大模型的边缘原生服务系统"
  (paper.oopus.info review of the FreeToken paper): §2 opening (two-level expert
  memory, slot per (layer, expert), GPU memory affects only performance),
  §2.2 (whole-layer double buffering), §2.4 (shared LRU expert cache),
  §2.5 (q* split, its equations, rounding and the exact merge), §2.6
  (device-side cache control), §2.7 (runtime cache reconfiguration, expert
  banks), Table 1 (measured B_P and B_H).
* [Overview] "FreeToken – 边缘原生的 MoE（混合专家）模型推理服务系统"
  (shshi.cn product page), section "FreeToken技术原理" items 1, 2 and 4.
* The gating function, the SwiGLU expert and the weight formats are not
  spelled out on the pages; the oracle takes the plain textbook definitions:
  softmax over all experts, top-k with the lowest index winning ties,
  renormalised over the k chosen; FFN(x) = W_d^T (silu(W_g^T x) * (W_u^T x));
  OCP MX v1.0 for e2m1 / e8m0, the e4m3 "fn" encoding, NVFP4 = e2m1 values
  with an e4m3 scale per 16 and an fp32 tensor scale.

Modules: ``moe`` (layer math), ``formats`` (decoders of the stored formats and
the bf16 rounding rule), ``lru`` (the expert-cache simulator), ``qsplit``
(the q* rule).  Every function is pinned by ``tests/test_oracle_*.py``.
"""
from . import formats, lru, moe, qsplit  # noqa: F401
