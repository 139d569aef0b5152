"""GB300-native sparse chunked-KV prefill and static-KV decode attention."""
