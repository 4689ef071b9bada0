"""Seeded token traces of the five workloads.

Each builder returns plain token arrays (int32) and sizes; the scenario logic
that feeds them to a cache lives with the callers.  The seed of workload i
(0-based, in the order tiny, few-shot, chat, agent tree, MLA) is 0x5EED + i and
is also the seed of its prefix hash.  Sibling branches are drawn with distinct
first tokens so that the designed tree shapes hold exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED0 = 0x5EED


@dataclass(frozen=True)
class Shape:
    q_heads: int
    kv_heads: int
    head_dim_k: int
    head_dim_v: int
    mla: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim_k))


GQA_TINY = Shape(4, 4, 64, 64)
GQA_32_8 = Shape(32, 8, 128, 128)
GQA_64_8 = Shape(64, 8, 128, 128)
MLA_128 = Shape(128, 1, 576, 512, mla=True)


def _rng(index: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([SEED0 + index, salt]))


def _distinct_firsts(rng, n, vocab, avoid=()):
    pool = np.setdiff1d(np.arange(vocab), np.asarray(list(avoid), dtype=np.int64))
    return rng.choice(pool, size=n, replace=False).astype(np.int32)


def _tokens(rng, n, vocab, first=None):
    t = rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)
    if first is not None and n > 0:
        t[0] = first
    return t


# ---------------------------------------------------------------- tiny (C1)
@dataclass
class TinyTrace:
    shape: Shape = GQA_TINY
    vocab: int = 1000
    seed: int = SEED0
    pool_slots: int = 2048
    max_new: int = 8
    system: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    prompts: list = field(default_factory=list)


def tiny(n_requests: int = 10) -> TinyTrace:
    """One shared 32-token system prompt + distinct 8..16-token questions."""
    rng = _rng(0)
    tr = TinyTrace()
    tr.system = _tokens(rng, 32, tr.vocab)
    firsts = _distinct_firsts(rng, n_requests, tr.vocab)
    for i in range(n_requests):
        qlen = int(rng.integers(8, 17))
        q = _tokens(rng, qlen, tr.vocab, first=firsts[i])
        tr.prompts.append(np.concatenate([tr.system, q]).astype(np.int32))
    return tr


def cyclic_prefixes(n_prefixes: int = 5, length: int = 64, vocab: int = 1000) -> list:
    """Prefixes A, B, C, ... of ``length`` tokens with distinct first tokens."""
    rng = _rng(0, salt=1)
    firsts = _distinct_firsts(rng, n_prefixes, vocab)
    return [_tokens(rng, length, vocab, first=f) for f in firsts]


def cyclic_order(n_prefixes: int, cycles: int, grouped: bool) -> list:
    """Request order as prefix indices: A..E repeated, or each prefix twice in a row."""
    if grouped:
        return [p for p in range(n_prefixes) for _ in range(cycles)]
    return [p for _ in range(cycles) for p in range(n_prefixes)]


# ------------------------------------------------------------ few-shot (C2)
@dataclass
class FewShotTrace:
    shape: Shape = GQA_32_8
    vocab: int = 32000
    seed: int = SEED0 + 1
    pool_slots: int = 1 << 21
    max_new: int = 128
    warm: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    questions: list = field(default_factory=list)

    def prompt(self, i: int) -> np.ndarray:
        return np.concatenate([self.warm, self.questions[i]]).astype(np.int32)


def few_shot(n_questions: int = 256, system_len: int = 512, n_examples: int = 5,
             example_len: int = 256, qmin: int = 32, qmax: int = 64,
             max_new: int = 128, batch_salt: int = 0) -> FewShotTrace:
    """512-token system prompt + 5 x 256-token examples, then distinct questions.

    ``batch_salt`` draws another batch of questions against the same warm prefix.
    """
    rng = _rng(1)
    tr = FewShotTrace(max_new=max_new)
    parts = [_tokens(rng, system_len, tr.vocab)]
    parts += [_tokens(rng, example_len, tr.vocab) for _ in range(n_examples)]
    tr.warm = np.concatenate(parts).astype(np.int32)
    qrng = _rng(1, salt=1 + batch_salt)
    # first tokens: one fixed permutation of the vocabulary, a disjoint slice
    # per batch, so a batch never matches another batch's cached questions
    perm = _rng(1, salt=100_000).permutation(tr.vocab).astype(np.int32)
    firsts = np.take(perm, np.arange(batch_salt * n_questions, (batch_salt + 1) * n_questions), mode="wrap")
    for i in range(n_questions):
        qlen = int(qrng.integers(qmin, qmax + 1))
        tr.questions.append(_tokens(qrng, qlen, tr.vocab, first=firsts[i]))
    return tr


# ---------------------------------------------------------------- chat (C3)
@dataclass
class ChatTrace:
    shape: Shape = GQA_32_8
    vocab: int = 32000
    seed: int = SEED0 + 2
    max_new: int = 128
    max_batch: int = 256
    pool_slots: int = 0
    user_turns: list = field(default_factory=list)  # [session][turn] -> tokens


def chat(n_sessions: int = 256, n_turns: int = 8, umin: int = 128, umax: int = 512,
         max_new: int = 128, pool_fraction: float = 0.75) -> ChatTrace:
    """Sessions growing turn by turn; the pool holds ``pool_fraction`` of the working set."""
    rng = _rng(2)
    tr = ChatTrace(max_new=max_new)
    firsts = _distinct_firsts(rng, n_sessions, tr.vocab)
    total = 0
    for s in range(n_sessions):
        turns = []
        for t in range(n_turns):
            ulen = int(rng.integers(umin, umax + 1))
            turns.append(_tokens(rng, ulen, tr.vocab, first=firsts[s] if t == 0 else None))
            total += ulen + max_new
        tr.user_turns.append(turns)
    tr.pool_slots = int(np.floor(pool_fraction * total))
    return tr


# ---------------------------------------------------------- agent tree (C4)
@dataclass
class AgentTrace:
    shape: Shape = GQA_64_8
    vocab: int = 32000
    seed: int = SEED0 + 3
    max_new: int = 256
    pool_slots: int = 65536
    root: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    branches: dict = field(default_factory=dict)  # path tuple -> tokens
    leaves: list = field(default_factory=list)    # list of path tuples

    def prompt(self, leaf) -> np.ndarray:
        parts = [self.root] + [self.branches[leaf[:i + 1]] for i in range(len(leaf))]
        return np.concatenate(parts).astype(np.int32)


def agent_tree(root_len: int = 2048, fanout: int = 4, depth: int = 3,
               branch_len: int = 256, max_new: int = 256) -> AgentTrace:
    rng = _rng(3)
    tr = AgentTrace(max_new=max_new)
    tr.root = _tokens(rng, root_len, tr.vocab)
    frontier = [()]
    for _ in range(depth):
        nxt = []
        for p in frontier:
            firsts = _distinct_firsts(rng, fanout, tr.vocab)
            for c in range(fanout):
                tr.branches[p + (c,)] = _tokens(rng, branch_len, tr.vocab, first=firsts[c])
                nxt.append(p + (c,))
        frontier = nxt
    tr.leaves = frontier
    return tr


# ----------------------------------------------------------------- MLA (C5)
@dataclass
class MLATrace:
    shape: Shape = MLA_128
    vocab: int = 32000
    seed: int = SEED0 + 4
    steps: int = 64
    pool_slots: int = 0
    shared: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    private: list = field(default_factory=list)

    def prompt(self, i: int) -> np.ndarray:
        return np.concatenate([self.shared, self.private[i]]).astype(np.int32)


def mla_long(batch: int = 128, shared_len: int = 4096, private_max: int = 28672,
             steps: int = 64) -> MLATrace:
    rng = _rng(4)
    tr = MLATrace(steps=steps)
    tr.shared = _tokens(rng, shared_len, tr.vocab)
    firsts = _distinct_firsts(rng, batch, tr.vocab)
    for i in range(batch):
        n = int(rng.integers(0, private_max + 1))
        tr.private.append(_tokens(rng, n, tr.vocab, first=firsts[i] if n else None))
    tr.pool_slots = shared_len + sum(len(p) for p in tr.private) + batch * steps
    return tr


# ------------------------------------------------------- multimodal (images)
@dataclass
class MultimodalTrace:
    """Questions about images, several per image, arriving interleaved.
    Images are raw bytes; a prompt is system + the image's key run + question,
    where the caller turns an image into keys with its own function (the
    product's rc_image_key, or the oracle's), so neither side's inputs come
    from the other."""
    shape: Shape = GQA_32_8
    vocab: int = 32000
    seed: int = SEED0 + 5
    max_new: int = 32
    image_tokens: int = 576
    pool_slots: int = 0
    system: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    images: list = field(default_factory=list)      # bytes
    questions: list = field(default_factory=list)   # (image index, tokens), arrival order

    def prompt(self, i: int, key_fn) -> np.ndarray:
        img, q = self.questions[i]
        keys = np.asarray(key_fn(self.images[img], self.image_tokens), np.int32)
        return np.concatenate([self.system, keys, q]).astype(np.int32)


def multimodal(n_images: int = 24, per_image: int = 8, system_len: int = 50, qmin: int = 16, qmax: int = 48,
               image_bytes: int = 4096, image_tokens: int = 576, max_new: int = 32) -> MultimodalTrace:
    rng = _rng(5)
    tr = MultimodalTrace(max_new=max_new, image_tokens=image_tokens)
    tr.system = _tokens(rng, system_len, tr.vocab)
    tr.images = [rng.integers(0, 256, image_bytes, dtype=np.int64).astype(np.uint8).tobytes()
                 for _ in range(n_images)]
    qs = []
    for img in range(n_images):
        for _ in range(per_image):
            qs.append((img, _tokens(rng, int(rng.integers(qmin, qmax + 1)), tr.vocab)))
    order = rng.permutation(len(qs))
    tr.questions = [qs[int(i)] for i in order]
    per_req = system_len + image_tokens + qmax + max_new
    tr.pool_slots = int(per_req * len(qs))
    return tr
