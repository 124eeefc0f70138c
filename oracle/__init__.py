"""Plain, slow CPU oracle for the MLA latent-cache decode step (fp64, NumPy).

TEST INFRASTRUCTURE ONLY. Nothing in the library package ``mla_latent_kv_69_b300``
imports, links or calls anything here; only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py`` may use it. The oracle shares
no code, table or constant generator with the CUDA path: the two meet only in the
seeded input generator (``workloads.py``), which holds none of the method's
arithmetic.

Sources (web pages, cited by title and section):

* [A] "DeepSeek-V2 机制拆解：KV 缓存压缩 93.3% 是怎么做到的" (discosf.com)
  - §"长上下文推理的第一瓶颈：93.3% KV 缓存压缩从何而来": decode re-reads every
    previous token's K/V; MHA caches 2·n_h·d_h·l elements per token; MLA caches a
    d_c = 512 latent c_KV from which K and V are up-projected at attention time;
    W_UK can be absorbed into W_Q and W_UV into W_O; the cache equals GQA with
    2.25 groups.
  - §"解耦 RoPE 与 YaRN：128K 上下文是怎么扩出来的": RoPE is carried by an extra
    decoupled per-head query and a shared key of width d_h^R = 64, keeping the
    compressed path position-free; the cache grows by d_h^R·l.
* [B] "DeepSeek-V2: A Strong, Economical, and Efficient Mixture-of-Experts
  Language Model - 中文验证版" (ai-papers.xuzou.cn)
  - §"瓶颈": the cache formulas and the 128K / 60-layer / 6-bit arithmetic
    (≈3.4 GB at batch 1, ≈217 GB at batch 64).
  - §"方法适配": d_c = 512, decoupled RoPE key width 64, 2.25-group GQA equivalence.
  - §"计算设置": 128 attention heads, 60 layers, hidden size 5120.

Modules:

* ``mla_oracle`` — RoPE, the explicit (non-absorbed) MLA decode attention, the
  absorbed form used only as a cross-check, the log-sum-exp merge of partial
  results, and the cache-size arithmetic.
* ``fp8_e4m3`` — the e4m3 ("fn": finite, no infinities) codec written from the
  format definition, and the per-token amax/448 row quantiser.
* ``fp6_e2m3`` — the e2m3 (6-bit) codec, the per-64-element-group quantiser and the
  four-codes-in-three-bytes packing of the ~6-bit cache reading; no CUDA path uses it
  yet.
"""

from . import fp6_e2m3, fp8_e4m3, mla_oracle  # noqa: F401
