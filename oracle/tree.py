"""Draft-tree bookkeeping: depth, RoPE positions, ancestor mask and bitmask.

Source: "Advanced speculative decoding: tree drafts and EAGLE", section "Why
trees" and its mask and depth helpers: node i attends to every committed
prefix position, to the nodes on its path from the root and to itself, and sits
at position prefix length + depth, so siblings share a position.  The root (node 0, parent -1) is the token the
target gave in the previous step.

Representation used on both sides: ``parents`` int32 [N] with parents[0] = -1
and 0 <= parents[i] < i (topological order), N <= 64, so the visibility row
of node i fits a 64-bit word: bit j set <=> node j is i or an ancestor of i.

Pinned by: the 6x6 mask the page prints for parents [-1, 0, 0, 1, 1, 2]
(tests/golden/tree_mask_6.txt), by agreement between the brute-force
ancestor walk and the bitmask recurrence on random trees, by depth from the
parent recurrence equal to the walk's ancestor count (two separate code
paths), and, for
``static_tree``, by the node counts the page's exercise 1 answers (14 and 30
draft nodes for branching [2, 2, 1, 1] and [3, 3, 2]).
"""
import numpy as np

MAX_NODES = 64


def validate(parents):
    """Raise ValueError unless ``parents`` is a topologically ordered tree."""
    p = [int(v) for v in parents]
    if not p or len(p) > MAX_NODES:
        raise ValueError("tree must have 1..64 nodes")
    if p[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for i in range(1, len(p)):
        if not 0 <= p[i] < i:
            raise ValueError(f"parent of node {i} must be in [0, {i})")


def static_tree(branching):
    """Parent array of a static tree: every node at depth t - 1 has branching[t - 1] children
    ("Advanced speculative decoding: tree drafts and EAGLE", section "Exercises", exercise 1).
    Nodes are numbered depth by depth; node 0 is the root."""
    parents, level = [-1], [0]
    for b in branching:
        nxt = []
        for par in level:
            for _ in range(int(b)):
                nxt.append(len(parents))
                parents.append(par)
        level = nxt
    return np.asarray(parents, dtype=np.int32)


def depths(parents):
    """Depth of every node by the parent recurrence: the root is at depth 0 and every other node
    is one deeper than its parent (parents precede their children)."""
    validate(parents)
    d = np.zeros(len(parents), dtype=np.int64)
    for i in range(1, len(parents)):
        d[i] = d[int(parents[i])] + 1
    return d


def positions(parents, prefix_len):
    """RoPE position of each node: prefix_len + depth."""
    return int(prefix_len) + depths(parents)


def mask_matrix(parents):
    """Boolean [N, N] visibility matrix by brute force: row i marks every node met while walking
    from node i up to the root, node i included."""
    validate(parents)
    n = len(parents)
    m = np.zeros((n, n), dtype=bool)
    for i in range(n):
        j = i
        while j != -1:
            m[i, j] = True
            j = int(parents[j])
    return m


def anc_bits(parents):
    """uint64 [N]: bit j of entry i set <=> node j is node i or one of its ancestors."""
    validate(parents)
    out = []
    for i, p in enumerate(parents):
        bits = 1 << i
        if p != -1:
            bits |= out[int(p)]
        out.append(bits)
    return np.asarray(out, dtype=np.uint64)


def children(parents, node):
    """Children of ``node`` in ascending node index."""
    return [c for c in range(len(parents)) if int(parents[c]) == node]


def path_to(parents, node):
    """Nodes from the root down to ``node`` inclusive."""
    out = []
    j = int(node)
    while j != -1:
        out.append(j)
        j = int(parents[j])
    return out[::-1]
