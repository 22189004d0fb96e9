"""The five decode workloads and their seeded synthetic tensors.

Shapes follow the Llama-style decoder the megakernel pages talk about
(« 2 · Définition et généalogie », §2.3 and « Résumé exécutif », "Le problème":
Llama-1B decode at batch 1).  The exact sizes are the workload definitions
of this project:

  tiny                 2 layers, H 256, 4 q / 2 kv heads of 64, FFN 768, vocab 1024,
                       theta 1e4, untied, batch 1, KV context 64, 8 steps
  llama1b_ctx1024      16 layers, H 2048, 32 q / 8 kv heads of 64, FFN 8192,
                       vocab 128256, tied, theta 5e5, batch 1, context 1024, 128 steps
  llama1b_ctx8192      same shape, context 8192, 64 steps
  llama1b_b8_ragged    same shape, batch 8, per-sequence context U{128..4096}, 64 steps
  llama8b_ctx2048      32 layers, H 4096, 32 q / 8 kv heads of 128, FFN 14336,
                       vocab 128256, untied, theta 5e5, batch 1, context 2048, 64 steps
  tiny_b4_ragged       the tiny shape at batch 4, per-sequence context U{16..64}, 8 steps

Recipe (all seeded, counter-based, see synth.c):
  projection and embedding matrices  bf16(N(0, 0.02))
  RMSNorm gains                      bf16(1 + N(0, 0.02))
  KV cache                           bf16(N(0, 1)) at positions < ctx_b, zero beyond
  step-0 tokens                      uniform in [0, vocab)
  ragged contexts                    uniform in [128, 4096]
"""
import numpy as np

from . import kv_bf16, normal_bf16, uniform_i32

LLAMA1B = dict(n_layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
               ffn_dim=8192, vocab=128256, rms_eps=1e-5, rope_theta=500000.0,
               tie_embeddings=1)
LLAMA8B = dict(n_layers=32, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
               ffn_dim=14336, vocab=128256, rms_eps=1e-5, rope_theta=500000.0,
               tie_embeddings=0)
TINY = dict(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=768,
            vocab=1024, rms_eps=1e-5, rope_theta=10000.0, tie_embeddings=0)

WORKLOADS = {
    "tiny": dict(model=TINY, batch=1, ctx=64, steps=8),
    "llama1b_ctx1024": dict(model=LLAMA1B, batch=1, ctx=1024, steps=128),
    "llama1b_ctx8192": dict(model=LLAMA1B, batch=1, ctx=8192, steps=64),
    "llama1b_b8_ragged": dict(model=LLAMA1B, batch=8, ctx=(128, 4096), steps=64),
    "llama8b_ctx2048": dict(model=LLAMA8B, batch=1, ctx=2048, steps=64),
    # small batched parity case (the tensor-core projections of batch > 1)
    "tiny_b4_ragged": dict(model=TINY, batch=4, ctx=(16, 64), steps=8),
    # larger-batch mode (batch 32: tensor cores, 16 KB pages, accumulator
    # read back sixteen sequences at a time)
    "tiny_b32_ragged": dict(model=TINY, batch=32, ctx=(16, 64), steps=8),
    "llama1b_b32_ragged": dict(model=LLAMA1B, batch=32, ctx=(128, 4096), steps=64),
}
ORDER = ["tiny", "llama1b_ctx1024", "llama1b_ctx8192", "llama1b_b8_ragged", "llama8b_ctx2048"]

# tensor ids for the generator
T_EMBED, T_FINAL_NORM, T_LM_HEAD = 1, 2, 3
LAYER_KINDS = ["attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down"]
T_KCACHE, T_VCACHE, T_TOKENS0, T_CTX, T_STEP_TOKENS = 0xF00001, 0xF00002, 0xF00010, 0xF00011, 0xF00020

WEIGHT_STD = 0.02


def layer_tid(layer, kind):
    return 16 + 16 * layer + LAYER_KINDS.index(kind)


def contexts(name, seed=0):
    """Prefilled KV length per sequence."""
    w = WORKLOADS[name]
    if isinstance(w["ctx"], tuple):
        lo, hi = w["ctx"]
        return uniform_i32(seed, T_CTX, w["batch"], lo, hi)
    return np.full(w["batch"], w["ctx"], dtype=np.int32)


def max_ctx(name, seed=0, steps=None):
    """KV capacity: longest context plus the decode steps, rounded up to 64."""
    w = WORKLOADS[name]
    steps = w["steps"] if steps is None else steps
    need = int(contexts(name, seed).max()) + steps
    return (need + 63) // 64 * 64


def shapes(m):
    H, d, nq, nkv, F, V = (m["hidden"], m["head_dim"], m["n_q_heads"], m["n_kv_heads"],
                           m["ffn_dim"], m["vocab"])
    return {
        "attn_norm": (H,), "wq": (nq * d, H), "wk": (nkv * d, H), "wv": (nkv * d, H),
        "wo": (H, nq * d), "mlp_norm": (H,), "w_gate": (F, H), "w_up": (F, H),
        "w_down": (H, F),
    }


def make_model(m, seed=0, tie=None):
    """Random-init decoder weights as bf16 bit patterns (numpy uint16), PyTorch
    Linear layout [out, in].  Returns a dict: embed, final_norm, lm_head (None
    when tied) and layers[l][kind]."""
    tie = m["tie_embeddings"] if tie is None else tie
    H, V = m["hidden"], m["vocab"]
    shp = shapes(m)
    model = {
        "embed": normal_bf16(seed, T_EMBED, (V, H), 0.0, WEIGHT_STD),
        "final_norm": normal_bf16(seed, T_FINAL_NORM, (H,), 1.0, WEIGHT_STD),
        "lm_head": None if tie else normal_bf16(seed, T_LM_HEAD, (V, H), 0.0, WEIGHT_STD),
        "layers": [],
    }
    for l in range(m["n_layers"]):
        layer = {}
        for kind in LAYER_KINDS:
            mean = 1.0 if kind.endswith("norm") else 0.0
            layer[kind] = normal_bf16(seed, layer_tid(l, kind), shp[kind], mean, WEIGHT_STD)
        model["layers"].append(layer)
    return model


def make_kv(m, batch, mctx, ctx, seed=0):
    """(K, V) caches, [L][B][nkv][max_ctx][d] bf16 bits, prefilled below ctx[b]."""
    args = (m["n_layers"], batch, m["n_kv_heads"], mctx, m["head_dim"], ctx)
    return kv_bf16(seed, T_KCACHE, *args), kv_bf16(seed, T_VCACHE, *args)


def first_tokens(m, batch, seed=0):
    return uniform_i32(seed, T_TOKENS0, batch, 0, m["vocab"] - 1)


def step_tokens(m, batch, steps, seed=0):
    """Token ids for free-running (bench) steps: [steps][batch] uniform."""
    return uniform_i32(seed, T_STEP_TOKENS, steps * batch, 0, m["vocab"] - 1).reshape(steps, batch)
