"""Python restatement of the plan sizing rule, for bit-exact plan tests.

Mirrors the documented behaviour of pa_plan_create with both overrides set:
kernel shape (rows per warp, warp split, stage tokens), ring depth from the
shared-memory budget, schedule/merge resolution, grid, partial slots and
workspace layout.
"""

SMEM_TWO = 112 * 1024
SMEM_ONE = 226 * 1024
COUNTER_STRIDE = 32


def align(x, a):
    return (x + a - 1) // a * a


def kernel_shape(d):
    G = d["num_q_heads"] // d["num_kv_heads"]
    R = G * d["query_len"]
    nt = 1
    rw = 8 * nt
    wr = -(-R // rw)
    wt = 1 if wr >= 4 else 4 // wr
    mx = d["kv_dtype"] == 2  # MXFP4: 64-byte rows (head_dim 128), the FP8 path
    elt = 1 if d["kv_dtype"] in (0, 2) else 2
    rb = d["head_dim"] // 2 if mx else d["head_dim"] * elt
    tt = min(128, max(16, 32768 // (2 * rb)))
    tw = 2 if (d["kv_dtype"] in (0, 2) and d["head_dim"] == 128) else 1
    k = dict(R=R, G=G, nt=nt, rw=rw, wr=wr, wt=wt, ncw=wr * wt, rpad=wr * rw, elt=elt, rb=rb,
             tt=tt, tw=tw, bh=min(d["page_size"], tt), umma=False, rh=0)
    # more than 16 rows on dense decode: the tensor-memory consumer (two
    # softmax warpgroups of rh rows, 128-token stages), taken by AUTO
    # (BF16 caches with FP16 queries stay on the tile consumer)
    supported = d.get("sparse_topk", 0) == 0 and not mx and d.get("v_layout", 0) == 0 and R > (
        8 if d["head_dim"] == 256 else 16) and (
        d["head_dim"] == 128 or (d["kv_dtype"] == 0 and d["head_dim"] == 256)) and not (
        d["kv_dtype"] == 1 and d.get("q_dtype", 0) == 1)
    consumer = d.get("consumer", 0)
    if supported and consumer in (0, 2):
        four = R > 32 and 0 < d.get("max_context_len", 0) <= 16384
        rh = 16 if (R <= 32 or four) else 32
        nwg = 4 if four else 2
        k.update(umma=True, rh=rh, nwg=nwg, nt=2, rw=rh, wr=nwg, wt=4, ncw=8, rpad=-(-R // 8) * 8, tt=128,
                 bh=min(d["page_size"], 128))
    return k


def smem_total(d, k, ns, cluster, nq):
    stage = 2 * k["tt"] * k["rb"] + (1024 if d["scale_mode"] in (2, 3) else 0)
    off = ns * stage
    if k["umma"]:
        rn = k["nwg"] * k["rh"]
        off += (3 if d["kv_dtype"] == 0 else 2) * d["head_dim"] * rn  # Q operand
        off = align(off, 1024)
        off += (3 if d["kv_dtype"] == 0 else 2) * k["tt"] * 128 + 2048  # P^T slots, the ones operand
    elif cluster:
        off += align(k["rpad"] * d["head_dim"] * 4 + k["rpad"] * 8, 128)
    off += ns * 128 + ns * 16 + 32 + (128 if k["umma"] else 16) + 16
    if k["umma"]:
        off += 8 * 64 * 4  # per-row state
    off = align(off, 16)
    off += 64 + 8 * 32 + (0 if k["umma"] else align(k["wt"] * k["rpad"] * 8, 128))
    off = align(off, 16)
    off += nq * k["rpad"] * d["head_dim"] * 2  # Q ring: nq slots of BF16 query rows
    return stage, off + 1024


def plan(d):
    """Expected pa_plan_info fields for a descriptor dict with overrides set."""
    k = kernel_shape(d)
    two = not k["umma"] and k["ncw"] <= 4 and (d["head_dim"] <= 128 or d["kv_dtype"] == 0)
    ns, budget = 0, SMEM_TWO
    cl0 = d.get("sparse_topk", 0) > 0 or d.get("merge_mode", 0) == 2
    for attempt in range(0 if two else 1, 2):
        if ns >= 3:
            break
        budget = SMEM_TWO if attempt == 0 else SMEM_ONE
        for nq in ((1,) if k["umma"] else (2, 1)):
            stage, total0 = smem_total(d, k, 0, cl0, nq)
            ns = min(8, (budget - total0) // (stage + 144))
            if ns >= 3:
                break
    assert ns >= 2
    sm, cps = d["sm_count_override"], d["ctas_per_sm_override"]
    units = d["batch"] * d["num_kv_heads"]
    sched, merge, P = d.get("schedule", 0), d.get("merge_mode", 0), d.get("max_partitions", 0)
    if merge == 1:
        sched, P = 2, 1
    if merge == 2:
        sched = 2
    if sched == 0:
        sched = 2 if (d.get("sparse_topk", 0) > 0 and units <= sm * cps) else 1
    if sched == 2:
        if P == 0:
            p = sm * cps // units if units > 0 else 1
            p = max(1, min(16, p))
            mt = d.get("sparse_topk", 0) or d.get("max_context_len", 0)
            if mt > 0:
                p = min(p, -(-mt // k["tt"]))
            P = max(1, p)
            if merge == 2 and P < 2:
                P = 2
    else:
        P = 0
    if merge == 0:
        merge = 3 if sched == 1 else (1 if P == 1 else (2 if P <= 8 else 3))
    if sched == 2 and P == 1:
        merge = 1
    cluster = merge == 2
    _, smem = smem_total(d, k, ns, cluster, nq)
    grid = sm * cps if sched == 1 else units * P
    if units == 0:
        grid = 0
    if sched == 1:
        slots = 2 * grid
    elif P > 1 and not cluster:
        slots = units * P
    else:
        slots = 0
    off = align(slots * k["rpad"] * d["head_dim"] * 4, 256)
    off = align(off + slots * k["rpad"] * 8, 256)
    if merge == 3 and slots > 0:
        off = align(off + units * COUNTER_STRIDE * 4, 256)
    if merge == 4:
        off = align(off + units * 16, 256)
    status = off
    off += 256
    return dict(merge_mode=merge, schedule=sched, num_partitions=P if sched == 2 else 0,
                stage_tokens=k["tt"], num_stages=ns, rows=k["R"], rows_per_warp=k["rw"],
                row_warps=k["wr"], token_warps=k["wt"], block_threads=32 * (4 * k["nwg"] + 2) if k["umma"] else (k["ncw"] + 1) * 32,
                grid=grid, cluster=P if cluster else 1, ctas_per_sm=cps, sm_count=sm,
                launches_per_call=2 if merge == 4 else 1, units=units, consumer=2 if k["umma"] else 1,
                smem_bytes=smem,
                workspace_bytes=off, partial_slots=slots, status_offset=status)
