"""gemm_launch_null: an empty kernel with the launch configuration of the
last call's main kernel (the identity null a benchmark times beside each
shape).  It must launch for every kernel family -- including the two-CTA
clusters and the 16-CTA clusters of the small-M kernel, whose cluster shapes
it reproduces -- leave C untouched, and refuse when there is no kernel to
mirror."""
import pytest
import torch

import dense_gemm_transformer_gb300 as dg

pytestmark = pytest.mark.gpu


@pytest.fixture()
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


def test_null_before_any_call_is_invalid(h):
    with pytest.raises(dg.GemmError) as e:
        h.launch_null()
    assert e.value.status == 1  # GEMM_ERR_INVALID_VALUE


@pytest.mark.parametrize("mode,M,N,K,family,cluster", [
    ("fp32", 300, 260, 200, "simt", 0),
    ("tf32", 512, 512, 256, "tc", 1),
    ("bf16", 2048, 2048, 256, "tc", 2),      # CTA pairs: clusters of 2
    ("bf16", 4, 1536, 8960, "skinny", 16),   # small M: clusters of 16 K slices
])
def test_null_mirrors_each_family(h, mode, M, N, K, family, cluster):
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    A = torch.randn(M, K, device="cuda").to(dt)
    B = torch.randn(K, N, device="cuda").to(dt)
    C = torch.empty(M, N, device="cuda")
    s = torch.cuda.Stream()
    h.run(A, B, C, mode=mode, stream=s)
    plan = h.plan()
    assert plan["family"] == family
    if cluster:
        assert plan["cluster"] == cluster
    before = C.clone()
    for _ in range(5):
        h.launch_null(s)
    assert h.check_device(s) == 0
    assert torch.equal(C, before)  # the null kernel touches no memory


def test_null_after_a_call_without_a_kernel_is_invalid(h):
    A = torch.randn(8, 8, device="cuda")
    C = torch.empty(8, 8, device="cuda")
    h.run(A, A, C, mode="fp32")
    h.launch_null()
    h.run(A, A, C, mode="fp32", alpha=0.0, beta=1.0)  # C = beta C: no GEMM kernel
    with pytest.raises(dg.GemmError):
        h.launch_null()
    torch.cuda.synchronize()
