"""B300-native forward of a token-choice top-k Mixture-of-Experts FFN layer."""
