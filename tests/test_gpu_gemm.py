"""The bf16 tcgen05 GEMM main loop against a plain fp32 product of the same
bf16 operands (C = A·Bᵀ), over tile-aligned, ragged and small shapes."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,bn,mt", [
    (128, 256, 64, 256, 1),        # one tile, one k-block
    (256, 512, 1024, 256, 1),      # several tiles and stages
    (300, 260, 192, 128, 1),       # ragged M and N
    (32, 6144, 4096, 128, 1),      # decode-shaped (M = 32)
    (1000, 768, 768, 256, 1),      # ragged M, N multiple of 256 with K 768
    (4096, 2304, 768, 256, 1),     # many tiles per CTA (persistent loop, accumulator ping-pong)
    # CTA pairs: a 256-row tile over two CTAs, each staging half of the weight tile
    (256, 256, 64, 256, 2),        # one pair tile, one k-block
    (300, 512, 1024, 256, 2),      # 3 row blocks: the second pair's odd CTA lies wholly past M
    (300, 768, 8192, 256, 2),      # the same with long K
    (1000, 768, 4096, 256, 2),     # ragged last block (104 rows), K of the Wo shape
    (1000, 512, 8192, 256, 2),     # 8 row blocks, the last one ragged
    (2048, 7168, 4096, 256, 2),    # 56 MB weight panel: grouped raster, several tiles per cluster
    (4096, 4096, 256, 256, 2),     # 16 x 16 pair tiles with four k-blocks each: short main loops
    (4096, 1280, 14336, 256, 2),   # 16 pair tiles x 5 column tiles over 76 clusters, K of the W2 shape
])
def test_gemm_bf16_matches_fp32_product(M, N, K, bn, mt):
    from causal_gqa_attention_rmsnorm_gb300 import binding
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    B = (0.05 * torch.randn(N, K, generator=g)).to(torch.bfloat16).cuda()
    C = binding.tbx_gemm_bf16(A, B, bn=bn, mt=mt)
    torch.cuda.synchronize()
    ref = A.double() @ B.double().T
    err = (C.double() - ref).abs().max().item()
    scale = ref.abs().max().item()
    # fp32 accumulation of K products: rounding ~ K·2^-24·max|a·b|
    assert err <= 1e-4 * max(scale, 1.0), (err, scale)
