"""Batch invariance of the layer: a token's output does not depend on the
other tokens of the batch.

The pages' point is train/rollout consistency: the same token must get the
same numbers whether it is scored in a large training batch or generated in
a small decode batch (NeMo RL FP8 article: token-mult-prob-error).  Every step of the
path here is per token or per (token, slot) pair with a fixed summation
order -- the router logits, top-k, the rotations, each output element of the
grouped GEMMs (the K order of a tile does not depend on how many tokens the
tile holds), and the slot-ordered combine -- so the forward output of a
token is bit-identical across batch sizes and chunk sizes.

Checked on the Kimi-K2-shaped INT4 layer: the first T tokens of the
T = 8192 batch, run alone for T = 1, 8, 64, 512, give the same Y rows bit
for bit.  The consistency measure of the pages is then reported through a
synthetic FP32 head: token-mult-prob-error = exp(mean |logp_a - logp_b|)
over the tokens, which is exactly 1 for identical outputs.
"""
import numpy as np
import pytest
import torch

from precision_moe_adapter_gb300 import build, pmoe
from precision_moe_adapter_gb300 import inputs as gi
from precision_moe_adapter_gb300.layer import DeviceLayer

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def forward_rows(cfg, w13, s13, w2, s2, Wr, bias, Su, Sd, X, C):
    L = DeviceLayer(cfg, w13, s13, w2, s2, Wr=Wr, bias=bias, S_up=Su, S_down=Sd)
    rt = L.new_routing()
    Xd = torch.from_numpy(np.ascontiguousarray(X)).view(torch.int16).cuda()
    L.route(Xd, rt)
    L.permute(rt)
    Y = torch.empty_like(Xd)
    L.forward(Xd, rt, Y, C=C, mode=pmoe.MODE_FUSED)
    torch.cuda.synchronize()
    assert L.status() == pmoe.PMOE_OK
    out = Y.cpu().numpy().view(np.uint16).copy(), rt.idx.cpu().numpy().copy()
    del L
    torch.cuda.empty_cache()
    return out


def token_mult_prob_error(Ya, Yb, seed=0, vocab=4096):
    """exp(mean_t |log p_a(y_t) - log p_b(y_t)|) through a synthetic FP32
    head W [d, vocab]; y_t is the head's argmax under a."""
    bf = lambda h: (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((Ya.shape[1], vocab)) * 0.02).astype(np.float32).astype(np.float64)

    def logp(Y):
        z = bf(Y) @ W
        z -= z.max(axis=1, keepdims=True)
        return z - np.log(np.exp(z).sum(axis=1, keepdims=True))

    la, lb = logp(Ya), logp(Yb)
    y = la.argmax(axis=1)
    t = np.arange(len(y))
    return float(np.exp(np.mean(np.abs(la[t, y] - lb[t, y]))))


def test_token_outputs_do_not_depend_on_the_batch():
    build.build()
    pmoe.lib()
    cfg = gi.CONFIGS["kimi_k2"]
    X = gi.gen_x(cfg)
    w13, s13, w2, s2 = gi.gen_weights(cfg)
    Wr, bias = gi.gen_router(cfg)
    Su, Sd = gi.gen_adapter_params(cfg)
    Y_full, idx_full = forward_rows(cfg, w13, s13, w2, s2, Wr, bias, Su, Sd, X, cfg.C)
    for T in (1, 8, 64, 512):
        sub = cfg.with_(T=T)
        for C in (8, cfg.C):
            Y, idx = forward_rows(sub, w13, s13, w2, s2, Wr, bias, Su, Sd, X[:T], C)
            assert np.array_equal(idx, idx_full[:T]), (T, C)
            assert np.array_equal(Y, Y_full[:T]), (T, C)
            assert token_mult_prob_error(Y_full[:T], Y) == 1.0
