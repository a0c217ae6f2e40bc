"""The benchmark's flop counts (CPU): the per-launch counts that the roofline
uses add up, over one step's launches, to the per-step layer figures."""

import pytest

import bench


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_per_launch_counts_add_up_to_the_step(name):
    w = bench.WORKLOADS[name]
    L, D, H, Hkv, U = w["L"], w["D"], w["H"], w["Hkv"], w["U"]
    attn, proj = bench.layer_flops(L, D, H, Hkv)  # 7 product-units of 2 (L^2/2) H d
    nch = H // U
    f = lambda k: bench.kernel_flops(k, w)
    # The forward kernel runs the layer figure's 2 forward products; the two
    # backward kernels execute 3 + 4 products (S and dP recomputed in the dQ
    # kernel), against the figure's 5 backward products.
    assert nch * f("attn_fwd") == pytest.approx(attn * 2 / 7)
    assert nch * (f("attn_bwd_dq") + f("attn_bwd_dkdv")) == pytest.approx(attn * 7 / 7)
    # Projections, when every chunk emits its K/V rows (U >= g): forward QKV
    # and O projection; backward dO, dWo, dWqkv and dx, the last two counted
    # once although the kernels run a high and a low bf16 half.
    if U >= H // Hkv:
        fwd = nch * (f("qkv_gemm") + f("oproj_gemm"))
        bwd = nch * (f("do_gemm") + f("dwo_gemm") + (f("dwqkv_gemm") + f("dx_gemm")) / 2)
        assert fwd + bwd == pytest.approx(proj)
