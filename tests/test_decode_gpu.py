"""Recurrent decoding (mc_decode_step): run token by token from empty caches, it
must reproduce the oracle's forward -- y for every token and the cached segment
states -- for every aggregation.

Pages cited:
  [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
  [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
           (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
"""
import numpy as np
import pytest
import torch

import memory_caching_linear_gb300 as mcl
import oracle
from mc_inputs import GRM, MEAN, RESIDUAL, SOUP, SSC, make_inputs
from ssc_valid import check_y_over_valid_sets, seg_starts

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from memory_caching_linear_gb300 import build
    build.build()
    mcl.load_library()


def decode_all(q, k, v, u, C, mode, topk, n_max):
    B, H, L, d = q.shape
    qd, kd, vd, ud = (x.cuda() if x is not None else None for x in (q, k, v, u))
    cache = mcl.DecodeCache(B, H, d, C, n_max)
    ys = []
    for t in range(L):
        tok = [x[:, :, t, :].contiguous() if x is not None else None for x in (qd, kd, vd, ud)]
        ys.append(mcl.mc_decode_step(cache, *tok, mode, topk).float().cpu())
    torch.cuda.synchronize()
    assert mcl.mc_check_device() == mcl.MC_OK
    return torch.stack(ys, 2).numpy(), cache


@pytest.mark.parametrize("mode,topk", [(RESIDUAL, 0), (GRM, 0), (SOUP, 0), (SSC, 2), (SSC, 4), (MEAN, 0)])
@pytest.mark.parametrize("d,C,L,dtype", [(64, 128, 512, "bf16"), (32, 48, 200, "f32"), (128, 256, 768, "bf16"),
                                         # 64 segments: the last token fills the 64th and last cache slot,
                                         # so reads near the end go over 63 cached states
                                         (128, 16, 1024, "bf16")])
def test_decode_reproduces_the_forward(mode, topk, d, C, L, dtype):
    q, k, v, u = make_inputs(1, 2, L, d, 17 + d + C, dtype)
    N = (L + C - 1) // C
    ref = oracle.forward(q, k, v, u, C, mode, topk)
    # the post-training average needs no router input
    y, cache = decode_all(q, k, v, None if mode == MEAN else u, C, mode, topk, n_max=min(N + 1, 64))
    yref = ref["y"]
    if mode == SSC and 0 < topk < N - 1:
        # near-ties in fp32 may rank either way: each such token must match the oracle
        # on one of its valid top-k selections
        ntie = check_y_over_valid_sets(
            y, q, k, v, u, seg_starts(L, C), topk, ref,
            lambda sel: oracle.forward(q, k, v, u, C, SSC, topk, given_sel=sel)["y"], TOL[dtype])
        print(f"near-tie tokens checked against their valid selections: {ntie}")
    else:
        err = np.abs(y - yref).max() / np.abs(yref).max()
        assert err <= TOL[dtype], err
    done = L // C  # segments completed by the last token
    st = cache.states[:, :, :done].cpu().numpy()
    serr = np.abs(st - ref["states"][:, :, :done]).max() / np.abs(ref["states"]).max()
    assert serr <= TOL["f32"], serr  # fp32 sums of the exact inputs


def test_decode_rejects_a_full_cache():
    q = torch.zeros(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    cache = mcl.DecodeCache(1, 1, 64, 16, n_max=2)
    cache.t = 32  # segment 2 does not fit in two slots
    with pytest.raises(mcl.MCError) as e:
        mcl.mc_decode_step(cache, q, q, q, q, GRM)
    assert e.value.status == mcl.MC_ERR_SHAPE
