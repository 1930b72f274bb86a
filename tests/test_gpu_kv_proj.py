"""GPU parity of ple_kv_proj (tcgen05 GEMM) against the oracle's float64
matmul, on tile-aligned and ragged shapes (M tails, N not a multiple of the
256-wide tile, K not a multiple of the 64-wide k-block), the tiny workload's
512 -> 2 x 1024 shape, and the 8k-prefill shape 8192 x 2048 -> 2 x 4096 in the
launch configuration the benchmark times (sampled rows through the oracle,
every row against cuBLAS as a library cross-check), for each kernel variant."""

import numpy as np
import pytest
import torch

from oracle import kv_proj as oracle_kv_proj

from _helpers import assert_close, bits, dev_err_word
from hashed_gram_embedding_gb300 import _lib

pytestmark = pytest.mark.gpu


def rand_bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("M,E,C", [(512, 512, 1024), (1, 64, 16), (129, 200, 48), (300, 2048, 4096),
                                   (1000, 128, 128), (257, 72, 112), (128, 64, 128)])
def test_kv_proj_matches_oracle(M, E, C):
    emb = rand_bf16((M, E), 0.5, M + E)
    w = rand_bf16((2 * C, E), 0.05, C + 7)
    kv = torch.full((M, 2 * C), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_kv_proj(emb.cuda(), w.cuda(), kv, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle_kv_proj(bits(emb), bits(w))
    assert_close(bits(kv), ref, what=f"kv {M}x{E}x{2*C}")


def test_kv_proj_is_deterministic_and_leaves_other_memory_alone():
    M, E, C = 700, 256, 320
    emb = rand_bf16((M, E), 1.0, 1).cuda()
    w = rand_bf16((2 * C, E), 0.05, 2).cuda()
    big = torch.full((M + 2, 2 * C), 7.0, dtype=torch.bfloat16, device="cuda")
    kv = big[1:M + 1]
    _lib.ple_kv_proj(emb, w, kv)
    first = kv.clone()
    _lib.ple_kv_proj(emb, w, kv)
    torch.cuda.synchronize()
    assert torch.equal(first, kv)
    assert torch.all(big[0] == 7.0) and torch.all(big[M + 1] == 7.0)


def test_kv_proj_prefill_8k_shape():
    M, E, C = 8192, 2048, 4096
    g = torch.Generator(device="cuda").manual_seed(11)
    emb = (torch.randn((M, E), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    w = (torch.randn((2 * C, E), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    kv = torch.empty((M, 2 * C), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_kv_proj(emb, w, kv, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    edges = [0, 1, 127, 128, 129, 255, 256, 4095, 4096, 8000, 8190, 8191]
    rest = np.setdiff1d(np.arange(M), edges)
    rows = np.concatenate([edges, np.random.default_rng(0).choice(rest, 2048, replace=False)])
    ref = oracle_kv_proj(bits(emb[torch.from_numpy(rows).cuda()]), bits(w))
    assert_close(bits(kv)[rows], ref, what="kv 8192x2048x8192 sampled rows")
    # all rows against cuBLAS (library cross-check, fp32 accumulate)
    lib_ref = (emb.float() @ w.float().T).to(torch.bfloat16)
    assert_close(bits(kv), bits(lib_ref), what="kv vs cuBLAS")


@pytest.mark.parametrize("mode", ["single", "pair", "pair-nosplit", "pair-epi4", "pair-epi8"])
@pytest.mark.parametrize("M,E,C", [(512, 512, 1024), (300, 2048, 4096), (129, 200, 48),
                                   (257, 72, 112), (1000, 128, 128)])
def test_kv_proj_kernel_variants(M, E, C, mode, monkeypatch):
    """Each kernel variant -- one CTA per 128 x 256 tile, CTA pairs with
    cta_group::2 MMAs over 256 x 256 tiles (with and without the last round
    split into 128-column halves; with 4 or 8 epilogue warps) -- gives the
    oracle's result, ragged edges included."""
    monkeypatch.setenv("PLE_KVPROJ_MODE", mode.split("-")[0])
    monkeypatch.setenv("PLE_KVPROJ_SPLIT", "0" if mode.endswith("nosplit") else "1")
    if "epi" in mode:
        monkeypatch.setenv("PLE_KVPROJ_EPI", mode[-1])
    emb = rand_bf16((M, E), 0.5, M + E)
    w = rand_bf16((2 * C, E), 0.05, C + 7)
    kv = torch.full((M, 2 * C), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_kv_proj(emb.cuda(), w.cuda(), kv, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(bits(kv), oracle_kv_proj(bits(emb), bits(w)), what=f"kv {mode} {M}x{E}x{2*C}")


@pytest.mark.parametrize("mode", ["single", "pair", "pair-nosplit", "pair-epi8"])
def test_kv_proj_variants_prefill_8k_against_cublas(mode, monkeypatch):
    monkeypatch.setenv("PLE_KVPROJ_MODE", mode.split("-")[0])
    monkeypatch.setenv("PLE_KVPROJ_SPLIT", "0" if mode.endswith("nosplit") else "1")
    if "epi" in mode:
        monkeypatch.setenv("PLE_KVPROJ_EPI", mode[-1])
    M, E, C = 8192, 2048, 4096
    g = torch.Generator(device="cuda").manual_seed(12)
    emb = (torch.randn((M, E), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    w = (torch.randn((2 * C, E), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    kv = torch.empty((M, 2 * C), dtype=torch.bfloat16, device="cuda")
    err = dev_err_word()
    _lib.ple_kv_proj(emb, w, kv, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    lib_ref = (emb.float() @ w.float().T).to(torch.bfloat16)
    assert_close(bits(kv), bits(lib_ref), what=f"kv {mode} vs cuBLAS")
