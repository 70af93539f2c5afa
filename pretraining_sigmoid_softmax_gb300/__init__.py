"""GB300-native fine-grained Mixture-of-Experts layer (forward and backward) for LLM
pretraining: sigmoid or softmax top-k routing, token permutation, SwiGLU experts as
tcgen05 grouped GEMMs, gate-weighted combine and the aux-loss-free bias update."""
from .configs import CONFIGS, MoEConfig  # noqa: F401
