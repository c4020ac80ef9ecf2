"""The five decode-attention workloads and the PCP prefill workload, with their sizes.

Shapes follow the pages' workloads: a toy GQA case, a Llama-8B-like GQA layer
(32 query heads over 8 KV heads, head_dim 128), and three MLA cases with one
shared 576-wide latent (512 latent + 64 RoPE) whose first 512 columns are the
values (the absorbed-MLA reading).  The mixed-length case stands in for the
agentic long-context trace with a ~67K median input that the DCP benchmark on
the Kimi K2.6 page uses; the trace itself is not available, so its lengths are
drawn lognormal around that median.
"""

import math

# dtype names used across the repo: "f32", "bf16", "fp8" (e4m3fn)
CONFIGS = {
    # GQA decode toy: fp32, everything tiny so the oracle finishes instantly.
    "gqa_toy": dict(
        index=1, layout="gqa", B=1, Tq=1, Hq=4, Hkv=1, Dk=64, Dv=64,
        lengths=("fixed", 256), N=2, I=1, block_size=16,
        q_dtype="f32", kv_dtype="f32", out_dtype="f32",
        softmax_scale=1.0 / math.sqrt(64),
    ),
    # GQA decode, Llama-8B-like layer.
    "gqa_llama8b": dict(
        index=2, layout="gqa", B=32, Tq=1, Hq=32, Hkv=8, Dk=128, Dv=128,
        lengths=("fixed", 8192), N=4, I=1, block_size=16,
        q_dtype="bf16", kv_dtype="bf16", out_dtype="bf16",
        softmax_scale=1.0 / math.sqrt(128),
    ),
    # MLA decode, bf16 latent cache, 32K context for every request.
    "mla_bf16_32k": dict(
        index=3, layout="mla", B=64, Tq=1, Hq=128, Hkv=1, Dk=576, Dv=512,
        lengths=("fixed", 32768), N=8, I=64, block_size=64,
        q_dtype="bf16", kv_dtype="bf16", out_dtype="bf16",
        softmax_scale=1.0 / math.sqrt(192),
    ),
    # MLA decode, FP8 latent cache, mixed long contexts (median 67K).
    "mla_fp8_mixed": dict(
        index=4, layout="mla", B=16, Tq=1, Hq=128, Hkv=1, Dk=576, Dv=512,
        lengths=("lognormal", 67 * 1024, 0.75, 4096, 200 * 1024), N=8, I=1,
        block_size=64, q_dtype="bf16", kv_dtype="fp8", out_dtype="bf16",
        softmax_scale=1.0 / math.sqrt(192),
    ),
    # MLA, a single 1M-token request with 4 causal query tokens per step.
    "mla_fp8_1m": dict(
        index=5, layout="mla", B=1, Tq=4, Hq=128, Hkv=1, Dk=576, Dv=512,
        lengths=("fixed", 1 << 20), N=8, I=1, block_size=64,
        q_dtype="bf16", kv_dtype="fp8", out_dtype="bf16",
        softmax_scale=1.0 / math.sqrt(192),
    ),
    # Prefill under PCP x DCP (the head-tail partition and causal prefill
    # path): a 2K-token chunk on top of a 64K cached context (the chunk and
    # context of the pages' prefill-overhead figure), Llama-8B-like GQA layer,
    # 4 DCP ranks holding the KV, 4 PCP ranks splitting the chunk, 64-token
    # pages (as the MLA configs).  Tq is the chunk; every request's last Tq
    # tokens are the new ones.
    "gqa_prefill_64k": dict(
        index=6, layout="gqa", B=2, Tq=2048, Hq=32, Hkv=8, Dk=128, Dv=128,
        lengths=("fixed", 64 * 1024 + 2048), N=4, I=1, block_size=64, pcp=4,
        q_dtype="bf16", kv_dtype="bf16", out_dtype="bf16",
        softmax_scale=1.0 / math.sqrt(128),
    ),
    # Sparse (top-k) MLA decode: config 4's mixed contexts, 4 query tokens per
    # request (an MTP-style step), each attending to 2,048 selected tokens
    # (the sparse-MLA selection size of the GLM-5.3 page), candidates from a
    # seeded synthetic indexer.
    "mla_fp8_sparse_2k": dict(
        index=7, layout="mla", B=16, Tq=4, Hq=128, Hkv=1, Dk=576, Dv=512,
        lengths=("lognormal", 67 * 1024, 0.75, 4096, 200 * 1024), N=8, I=1,
        block_size=64, topk=2048, q_dtype="bf16", kv_dtype="fp8", out_dtype="bf16",
        softmax_scale=1.0 / math.sqrt(192),
    ),
}

CONFIG_ORDER = ["gqa_toy", "gqa_llama8b", "mla_bf16_32k", "mla_fp8_mixed", "mla_fp8_1m"]


def config(name, **overrides):
    """A copy of a named config, with fields overridden (e.g. a smaller B or L)."""
    c = dict(CONFIGS[name])
    c["name"] = name
    for k, v in overrides.items():
        if k == "L":
            c["lengths"] = ("fixed", int(v))
        else:
            c[k] = v
    return c
