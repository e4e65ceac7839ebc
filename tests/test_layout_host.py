"""Host checks of the kernels' index arithmetic against the plans the
library returns (no CUDA call): for every plan, the float4 slots a CTA or a
lane group can touch fit the shared memory or registers the plan sizes, at
every row alignment, and the slices of a cluster cover the row exactly.
The layouts restated here are the ones the kernel sources document: a
segment starting at float offset `pad` (0..3) of a 16-byte line spans
ceil((pad + len) / 4) float4s."""
import pytest

import entropy_bounded_softmax_gb300 as cs

GB300 = dict(sm_count=152, smem_per_block_optin=232448, smem_per_sm=233472,
             max_cluster=16)


def float4s(pad, length):
    return (pad + length + 3) // 4


@pytest.mark.parametrize("batch", [1, 7, 32, 4096])
@pytest.mark.parametrize("C", [1, 3, 513, 4099, 8193, 32000, 50001, 131072,
                               464000, 850000])
def test_backward_cluster_slices(batch, C):
    st, p = cs.cs_plan_backward_host(batch, C, None, *GB300.values())
    assert st == 0
    p = p.as_dict()
    if p["variant"] != 2:
        return
    n, L = p["cluster_size"], p["slice_len"]
    covered = sum(max(0, min(L, C - r * L)) for r in range(n))
    assert covered == C
    for pad in range(4):
        q4 = float4s(pad, min(L, C))
        # shared memory: a 512-byte header, then slice_len / 4 + 1 float4s
        # of p (and as many of g when both are staged).
        assert q4 <= L // 4 + 1
        need = 512 + (L // 4 + 1) * 16 * p["staged_tensors"]
        assert need <= p["smem_bytes"] <= GB300["smem_per_block_optin"]


@pytest.mark.parametrize("C", [1, 2, 3, 5, 31, 64, 127, 257, 511, 512])
def test_backward_rowgroup_slots(C):
    st, p = cs.cs_plan_backward_host(100, C, None, *GB300.values())
    assert st == 0
    p = p.as_dict()
    assert p["variant"] == 1
    G, E = p["lanes_per_row"], p["elems_per_lane"] // 4
    for pad in range(4):
        assert float4s(pad, C) <= G * E


@pytest.mark.parametrize("S", [1, 2, 5, 64, 511, 512, 513, 1017, 1018, 1024,
                               1025, 4099, 57344])
@pytest.mark.parametrize("aligned", [0, 1])
def test_attention_slots(S, aligned):
    st, p = cs.cs_plan_attention_host(2, 2, S, aligned, None, 152, 232448,
                                      233472)
    assert st == 0
    p = p.as_dict()
    pads = [0] if aligned else range(4)
    if p["variant"] == 1:
        for pad in pads:
            assert float4s(pad, S) <= p["lanes_per_row"] * p["elems_per_lane"] // 4
    else:
        for pad in range(4):
            # 512-byte header, then (S + 6) / 4 + 1 float4s of the row.
            assert 512 + 16 * float4s(pad, S) <= p["smem_bytes"]
        assert p["smem_bytes"] <= 232448


@pytest.mark.parametrize("K", [1, 4, 5, 63, 64, 65, 128, 200, 256])
@pytest.mark.parametrize("D", [4, 64, 100])
def test_biencoder_smem(K, D):
    st, p = cs.cs_plan_biencoder_host(2, 300, K, D, 3, None, 232448)
    if st == 7:
        assert 4 * 2 * K * D > 200000      # keys and values alone too big
        return
    assert st == 0
    p = p.as_dict()
    G = p["lanes_per_row"]
    assert 16 * G >= K and (G == 1 or 8 * G < K) and p["elems_per_lane"] == 16
    R = p["threads_per_cta"] // G
    kp = (K + 3) // 4 * 4
    # every 4 x 4 block of a tile's scores has a thread
    assert (R // 4) * (kp // 4) <= p["threads_per_cta"]
    # scores rows: for G < 8 the stride is 4 G mod 32 (the rows of a
    # quarter-warp's 16-byte reads in different banks)
    ssw = kp + 4 if G >= 8 else kp + (4 * G - kp) % 32
    assert ssw >= kp and (G >= 8 or ssw % 32 == 4 * G % 32)
    if p["tensor_cores"]:
        # steps 1-2 only (keys, a query tile and its scores); step 3 on the
        # tensor cores
        assert K <= D <= 64 and p["staged_tensors"] == 2
        need = 4 * (D * kp + R * (D + 4) + R * ssw)
    else:
        need = 4 * (D * kp + K * D + R * (D + 4) + R * ssw)
    assert need == p["smem_bytes"] <= 232448
