"""Oracle for the plan-time tile configuration heuristic.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Restates the DeepGEMM
configuration heuristic ("Deep dive into DeepGEMM", blog.kumaling.xyz, panel
"Kernel Configuration Heuristic", step 2 "Performance Model") in the page's
order and notation:

  num_blocks      = ceil(M / BM) * ceil(N / BN)
  num_waves       = ceil(num_blocks / num_sms)
  wave_efficiency = num_blocks / (num_waves * num_sms)
  bytes_L2_AB     = K * (BM / cluster_N + BN / cluster_M) * sizeof(AB)
  bytes_local_AB  = K * (BM + BN) * sizeof(AB)
  bytes_TC        = K * (max(64, BM) + BN) * sizeof(AB) + BM * BN * sizeof(C)
  bytes_CD        = BM * BN * sizeof(C) * (2 if accumulating into C else 1)
  cycles_L2       = (bytes_L2_AB + bytes_CD) * num_blocks / BW_L2
  cycles_local    = (bytes_local_AB + bytes_TC + bytes_CD) * num_blocks / BW_local
  score           = max(cycles_local, cycles_L2) / wave_efficiency   (minimum wins)

Readings: BM and BN are the per-CTA block; a CTA pair (tcgen05 cta_group::2,
each CTA loading half of B) is the page's cluster 2 x 1, i.e. cluster_M = 2;
the candidate space is what the sm_103a kernel supports: BM = 128, BN in
{128, 256}, cluster_M in {1, 2}, cluster_N = 1; ties go to the larger block.
The bandwidths are whole-GPU bytes per SM cycle.
"""
from __future__ import annotations

from math import ceil

BW_L2 = 9000.0            # ~17 TB/s of TMA reads from L2 at ~1.9 GHz, measured on the listed workloads
BW_LOCAL_PER_SM = 256.0   # shared-memory-side bytes per cycle per SM


def score(M, N, K, BM, BN, cluster_m, cluster_n, sizeof_ab, sizeof_c, num_sms, accumulate=False,
          bw_l2=BW_L2, bw_local_per_sm=BW_LOCAL_PER_SM):
    num_blocks = ceil(M / BM) * ceil(N / BN)
    num_waves = ceil(num_blocks / num_sms)
    wave_efficiency = num_blocks / (num_waves * num_sms)
    bytes_l2_ab = K * (BM / cluster_n + BN / cluster_m) * sizeof_ab
    bytes_local_ab = K * (BM + BN) * sizeof_ab
    bytes_tc = K * (max(64, BM) + BN) * sizeof_ab + BM * BN * sizeof_c
    bytes_cd = BM * BN * sizeof_c * (2 if accumulate else 1)
    cycles_l2 = (bytes_l2_ab + bytes_cd) * num_blocks / bw_l2
    cycles_local = (bytes_local_ab + bytes_tc + bytes_cd) * num_blocks / (bw_local_per_sm * num_sms)
    return dict(num_blocks=num_blocks, num_waves=num_waves, wave_efficiency=wave_efficiency,
                bytes_l2_ab=bytes_l2_ab, bytes_local_ab=bytes_local_ab, bytes_tc=bytes_tc, bytes_cd=bytes_cd,
                cycles_l2=cycles_l2, cycles_local=cycles_local,
                score=max(cycles_local, cycles_l2) / wave_efficiency)


def choose(M, N, K, sizeof_ab, sizeof_c, num_sms):
    """(BN, cluster_M) of the lowest score; on a tie the larger BN, then the pair."""
    best = None
    for BN in (256, 128):
        for cm in (2, 1):
            if cm == 2 and M <= 128:
                continue  # a pair needs two 128-row blocks
            s = score(M, N, K, 128, BN, cm, 1, sizeof_ab, sizeof_c, num_sms)["score"]
            if best is None or s < best[0] * (1 - 1e-12):
                best = (s, BN, cm)
    return best[1], best[2]
