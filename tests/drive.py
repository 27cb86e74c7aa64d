"""Test helpers: replay a synth workload on the oracle's bookkeeping model."""
from oracle.cache import CacheModel


def oracle_run_ops(model, w, ops=None, names=None):
    names = {} if names is None else names
    for op in (w.ops if ops is None else ops):
        kind = op[0]
        if kind == "alloc":
            names[op[1]] = model.seq_alloc()
        elif kind == "fork":
            names[op[1]] = model.seq_fork(names[op[2]], op[3])
        elif kind == "append":
            model.append(names[op[1]], op[2])
        elif kind == "drop":
            model.drop(names[op[1]], op[2], op[3])
        elif kind == "repos":
            model.repos(names[op[1]], op[2], op[3], op[4])
        elif kind == "splice":
            model.splice(names[op[1]], op[2], op[3], op[4])
        elif kind == "flush":
            model.flush([names[op[1]]])
        elif kind == "compact":
            model.compact(names[op[1]])
        else:
            raise ValueError(kind)
    return names


def oracle_model(w):
    return CacheModel(w.n_pages, w.shape.page_size)
