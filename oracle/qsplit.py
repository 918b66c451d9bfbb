"""q* miss split -- [Review] §2.5 "核心公式：q* 带宽自适应策略".

The misses M of one layer step are split into F (filled into the GPU cache
over the host link) and C (evaluated where the weights live, outside the GPU),
q = |F|.  With B_P the pinned->device transfer bandwidth and B_H the host-side
expert bandwidth, the residual bandwidth is B_R = max(B_H - B_P, 0) (§2.5,
residual-bandwidth equation), the branch times are T_fill(q) = qS/B_P and
T_cpu(m-q) = (m-q)S/(B_H-B_P) (§2.5, branch-time equations), and equal times
give q* = m B_P / B_H (§2.5, balance equation).  q* is rounded half up
("四舍五入"), at least one expert is always filled, and as B_H falls to B_P
q* reaches m (§2.5, paragraph after the balance equation).
"""
import math


def residual_bandwidth(bw_fill: float, bw_host: float) -> float:
    """B_R = max(B_H - B_P, 0)."""
    return max(bw_host - bw_fill, 0.0)


def t_fill(q: float, S: float, bw_fill: float) -> float:
    """Time to move q experts of S bytes over the host link."""
    return q * S / bw_fill


def t_cpu(n: float, S: float, bw_fill: float, bw_host: float) -> float:
    """Time to evaluate n experts on the residual host bandwidth (inf when B_R = 0)."""
    br = residual_bandwidth(bw_fill, bw_host)
    return math.inf if br == 0.0 else n * S / br


def q_star_real(m: int, bw_fill: float, bw_host: float) -> float:
    """Unrounded balance point q* = m B_P / B_H (m when B_H <= B_P)."""
    if bw_host <= bw_fill:
        return float(m)
    return m * bw_fill / bw_host


def qsplit(m: int, bw_fill: float, bw_host: float) -> int:
    """Number of misses to fill: round-half-up of q*, clamped to [1, m]; 0 when m = 0."""
    if m <= 0:
        return 0
    if bw_host <= bw_fill:
        return m
    return qsplit_ratio(m, bw_fill / bw_host)


def qsplit_ratio(m: int, ratio: float) -> int:
    """Same rule given ratio = B_P / B_H directly (ratio >= 1 means fill every miss)."""
    if m <= 0:
        return 0
    if ratio >= 1.0:
        return m
    q = math.floor(m * ratio + 0.5)
    return min(m, max(1, q))
