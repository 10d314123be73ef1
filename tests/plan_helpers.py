"""Plan step lists shared by the plan tests (descriptions only, no arithmetic)."""
import random

import all_reduce_reduction_gb300 as ar


def builtin_steps(R, algo, K):
    """The two all-reduce algorithms as plan steps (buffer ids: b < R is
    in[b], R + r is out[r]), with R * K chunks."""
    steps = []
    if algo == "one_shot":
        for r in range(R):
            steps.append(dict(kind="reduce", rank=r, dst=R + r, srcs=list(range(R)),
                              cbeg=0, cend=R * K))
    else:
        for j in range(R):
            steps.append(dict(kind="reduce", rank=j, dst=R + j, srcs=list(range(R)),
                              cbeg=j * K, cend=(j + 1) * K))
        for r in range(R):
            for j in range(R):
                if j != r:
                    steps.append(dict(kind="copy", rank=r, dst=R + r, srcs=[R + j],
                                      cbeg=j * K, cend=(j + 1) * K))
    return steps


def random_steps(R, nchunks, nsteps, seed, copy_weight=1):
    """Random copy/reduce steps with plenty of cross-rank dependencies
    (copies are `copy_weight` times as likely as with the default mix)."""
    rng = random.Random(seed)
    steps = []
    for _ in range(nsteps):
        cb = rng.randrange(nchunks)
        ce = rng.randrange(cb + 1, nchunks + 1)
        kind = rng.choice(["copy"] * copy_weight + ["reduce", "reduce"])
        src_kind = rng.choice([0, 1])
        if kind == "copy":
            srcs = [src_kind * R + rng.randrange(R)]
        else:
            srcs = [src_kind * R + rng.randrange(R) for _ in range(rng.randint(1, R))]
        steps.append(dict(kind=kind, rank=rng.randrange(R), dst=R + rng.randrange(R), srcs=srcs,
                          cbeg=cb, cend=ce))
    return steps


def to_ops(steps, R):
    """Plan steps -> the library's ar_op structures."""
    ops = []
    for st in steps:
        buf = lambda b: (b // R, b % R)
        kind = ar.AR_OP_COPY if st["kind"] == "copy" else ar.AR_OP_REDUCE
        ops.append(ar.make_op(kind, st["rank"], buf(st["dst"]), [buf(b) for b in st["srcs"]],
                              st["cbeg"], st["cend"]))
    return ops
